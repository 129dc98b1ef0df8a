"""Benchmark of the MoE decode step (weight-streaming GB/s over the unique expert bytes).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--rows M]

One step = router GEMV + top-k, route, gate_up + down (one launch), finalize (moe_step,
four chained launches; five with MOE_FUSED_FFN=0) captured in a CUDA graph, on seeded
synthetic inputs of the workload's shapes. Between timed steps (untimed) a 512 MiB buffer
is written and another read, so every step streams its weights from HBM and finds no dirty
line of the flush in L2. Under torchrun each rank runs an independent replica (the step
has no cross-GPU exchange); the JSON line reports the sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "mxfp8_h7168_e256_k8_8rows"
METRIC = "MoE decode step weight GB/s (unique expert + shared + router bytes per step / step time)"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=HEADLINE)
    ap.add_argument("--rows", type=int, default=None)
    ap.add_argument("--experts", type=int, default=None, help="override E (smaller profiling cases)")
    ap.add_argument("--inter", type=int, default=None, help="override I and shared I (smaller profiling cases)")
    ap.add_argument("--swiglu-limit", type=float, default=None, help="clamped SwiGLU limit (default: plain SwiGLU)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    return ap.parse_args()


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _cfg(a):
    from moe_decode_step_router_gb300 import synth
    over = {}
    if a.rows is not None:
        over["M"] = a.rows
    if a.experts is not None:
        over["E"] = a.experts
    if a.inter is not None:
        over["I"] = over["I_sh"] = a.inter
    if a.swiglu_limit is not None:
        over["swiglu_limit"] = a.swiglu_limit
    return synth.config(a.config, **over)


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


def _cpu_baseline(cfg, inp, budget_s=20.0):
    """Time the oracle, as it stands, on whole rows of the same workload (bounded)."""
    import numpy as np
    import torch
    import oracle

    u16 = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)
    n = lambda t: None if t is None else t.detach().cpu().numpy()
    L = oracle.make_layer(cfg, inp["gs_a"])
    x16, wg16, r16, g16 = u16(inp["x"]), u16(inp["wg"]), u16(inp["residual"]), u16(inp["gamma"])
    bias = n(inp["bias"])
    E = cfg["E"]
    w13, w2 = [None] * E, [None] * E
    sh = lambda k: (n(inp[k][0][0]), n(inp[k][1][0]) if inp[k][1] is not None else None, float(inp[k][2][0]))
    sh13, sh2 = (sh("sh13"), sh("sh2")) if "sh13" in inp else (None, None)
    rows_done, t_total = 0, 0.0
    M = cfg["M"]
    for m in range(M):
        _, _, idx, _, _ = oracle.router(L, x16[m:m + 1], wg16, bias=bias)
        for e in idx.ravel():
            if w13[e] is None:
                w13[e] = (n(inp["w13"][0][e]), n(inp["w13"][1][e]) if inp["w13"][1] is not None else None,
                          float(inp["w13"][2][e]))
                w2[e] = (n(inp["w2"][0][e]), n(inp["w2"][1][e]) if inp["w2"][1] is not None else None,
                         float(inp["w2"][2][e]))
        t0 = time.perf_counter()
        oracle.step_rows(L, [m], x16, r16, g16, wg16, bias, w13, w2, sh13, sh2)
        t_total += time.perf_counter() - t0
        rows_done += 1
        if t_total > budget_s:
            break
    per_row = t_total / rows_done
    return per_row * M, rows_done


def _reference_arm(a):
    """The oracle as the reference implementation, on the same metric and workload."""
    import torch
    from moe_decode_step_router_gb300 import synth

    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    cfg = _cfg(a)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = synth.make_inputs(cfg, a.seed, device=dev)
    import numpy as np
    import oracle
    u16 = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)
    L = oracle.make_layer(cfg, inp["gs_a"])
    _, _, idx, _, _ = oracle.router(L, u16(inp["x"]), u16(inp["wg"]),
                                    bias=None if inp["bias"] is None else inp["bias"].cpu().numpy())
    n_active = len(np.unique(idx))
    ubytes = synth.unique_weight_bytes(cfg, n_active)
    per_step_budget = max(2.0, 60.0 / max(1, a.steps + a.warmup))
    times = []
    for i in range(a.warmup + a.steps):
        t, rows = _cpu_baseline(cfg, inp, budget_s=per_step_budget)
        if i >= a.warmup:
            times.append(t)
    t = sum(times) / len(times)
    val = ubytes / t / 1e9
    sample = "oracle rows timed until %.0f s per step, scaled to %d rows" % (per_step_budget, cfg["M"])
    line = {"metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": cfg["name"], "rows": cfg["M"], "unique_experts": n_active,
                       "unique_bytes": ubytes},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    a = _args()
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

    out = torch.zeros(M, H, dtype=torch.bfloat16, device=dev)
    res = inp["residual"].clone()
    M8 = -(-M // 8) * 8
    oq = torch.zeros(M8, H, dtype=torch.uint8, device=dev) if cfg["emit_next"] else None
    os_ = torch.zeros(M8, H // 32, dtype=torch.uint8, device=dev) if cfg["emit_next"] else None
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    args = layer.args(inp["x"], res, out, oq, os_)
    # warm the eager path once, then capture one graph of the whole step
    with torch.cuda.stream(stream):
        layer.step(inp["x"], res, out, oq, os_, stream=stream, args=args)
    stream.synchronize()
    if layer.status(stream) != 0:
        raise RuntimeError("device status %d after the first step" % layer.status(stream))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        layer.step(inp["x"], res, out, oq, os_, stream=stream, args=args)
    # L2 flush between timed steps: write one 512 MiB buffer, then read another, so that no
    # step input stays in the 129 MB L2 and no dirty line of the flush is left for the step
    # to write back (between two MoE layers of a decode loop L2 holds mostly clean lines).
    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(128 << 20, dtype=torch.float32, device=dev)
    flush_acc = torch.zeros((), dtype=torch.float32, device=dev)

    def flush_l2(v):
        flush_w.fill_(v)
        torch.sum(flush_r, dim=0, out=flush_acc)

    def one(timed_events=None):
        with torch.cuda.stream(stream):
            flush_l2(1)
            if timed_events:
                timed_events[0].record(stream)
            graph.replay()
            if timed_events:
                timed_events[1].record(stream)

    for _ in range(max(3, a.warmup)):
        one()
    stream.synchronize()
    clocks = Clocks(local)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0 = time.perf_counter()
    for i in range(a.steps):
        one(ev[i])
    stream.synchronize()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    step_ms = [s.elapsed_time(e) for s, e in ev]
    ms_step = _max_over_ranks(np.mean(step_ms), world, dev)
    st = layer.status(stream)
    if st != 0:
        raise RuntimeError("device status %d after the timed steps" % st)

    counts = layer.ws_tensor("expert_counts", torch.int32, (cfg["E"] + 1,)).cpu().numpy()
    n_active = int((counts[:cfg["E"]] > 0).sum())
    ubytes = synth.unique_weight_bytes(cfg, n_active)
    gbs = ubytes / (ms_step * 1e-3) / 1e9

    # ---- per-kernel timing of the two GEMMs, live, on the launching stream (routing of this step)
    v = layer.view
    ws_t = lambda name, dt, shp: layer.ws_tensor(name, dt, shp)
    perm = ws_t("perm", torch.int32, (M * cfg["k"] + M,))

    def gemm_time(fn, reps=max(10, a.steps // 2)):
        tt = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                flush_l2(2)
                e0.record(stream)
                fn()
                e1.record(stream)
            tt.append((e0, e1))
        stream.synchronize()
        return float(np.mean([s.elapsed_time(e) for s, e in tt]))

    q = layer.qw
    gu_ms = gemm_time(lambda: ms.moe_expert_gate_up(layer.d, q["w13"], q["sh13"], v.xq, v.xq_scales, v.xq_shared,
                                                    v.xq_shared_scales, perm, M, v.hq, v.hq_scales, layer.ws, stream))
    dn_ms = gemm_time(lambda: ms.moe_expert_down(layer.d, q["w2"], q["sh2"], v.hq, v.hq_scales, M, v.y_pairs,
                                                 layer.ws, stream))
    # the step runs both GEMMs as one launch unless MOE_FUSED_FFN=0
    fused = os.environ.get("MOE_FUSED_FFN", "1") != "0"
    ffn_ms = gemm_time(lambda: ms.moe_expert_ffn(layer.d, q["w13"], q["sh13"], q["w2"], q["sh2"], v.xq, v.xq_scales,
                                                 v.xq_shared, v.xq_shared_scales, perm, M, v.hq, v.hq_scales,
                                                 v.y_pairs, layer.ws, stream))

    def proj(fmt, rows, K):
        rb = 2 * K if fmt == 0 else (K if fmt == 1 else K // 2)
        rs = K // 32 if fmt in (1, 3) else (K // 16 if fmt == 2 else 0)
        return rows * (rb + rs) + (4 if fmt == 2 else 0)

    I, Ish = cfg["I"], cfg["I_sh"]
    gu_bytes = n_active * proj(cfg["w_fmt"], 2 * I, H) + (proj(cfg["sh_fmt"], 2 * Ish, H) if cfg["has_shared"] else 0)
    dn_bytes = n_active * proj(cfg["w_fmt"], H, I) + (proj(cfg["sh_fmt"], H, Ish) if cfg["has_shared"] else 0)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        peak, peak_src = 6800.0, "fallback"
    full_size = a.rows is None and a.experts is None and a.inter is None
    tr = _traffic_ratios() if full_size else {}

    def kern(part, nbytes, t_ms):
        key = cfg["name"] + "." + part
        return {"achieved": nbytes / (t_ms * 1e-3) / 1e9, "ms": t_ms, "algorithmic_bytes": nbytes,
                "traffic": tr[key] * nbytes if key in tr else None}

    # dominant kernel: the launch that runs the step's GEMMs, timed alone on the same routing
    if fused:
        dom, name = kern("ffn", gu_bytes + dn_bytes, ffn_ms), "k_expert_gemm(gate_up+down)"
    else:
        dom, name = kern("gate_up", gu_bytes, gu_ms), "k_expert_gemm(gate_up)"
    roofline = {"bound": "hbm", "kernel": name, "achieved": dom["achieved"], "peak": peak, "peak_source": peak_src,
                "unit": "GB/s", "frac": dom["achieved"] / peak, "traffic": dom["traffic"],
                "algorithmic_bytes": dom["algorithmic_bytes"], "ms": dom["ms"],
                "gate_up": kern("gate_up", gu_bytes, gu_ms), "down": kern("down", dn_bytes, dn_ms),
                "step_frac": gbs / peak}

    # ---- end to end through the C ABI with host buffers: H2D inputs, step, D2H output
    x_h = inp["x"].cpu().pin_memory()
    r_h = inp["residual"].cpu().pin_memory()
    o_h = torch.empty(M, H, dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty_like(inp["x"])
    e2e_args = layer.args(x_d, res, out, oq, os_)
    e2e = []
    for i in range(a.warmup + max(5, a.steps // 2)):
        with torch.cuda.stream(stream):
            flush_l2(3)
        stream.synchronize()
        t1 = time.perf_counter()
        with torch.cuda.stream(stream):
            x_d.copy_(x_h, non_blocking=True)
            res.copy_(r_h, non_blocking=True)
            layer.step(x_d, res, out, oq, os_, stream=stream, args=e2e_args)
            o_h.copy_(out, non_blocking=True)
        stream.synchronize()
        if i >= a.warmup:
            e2e.append(time.perf_counter() - t1)
    e2e_s = float(np.median(e2e))
    h2d = x_h.numel() * 2 + r_h.numel() * 2
    d2h = o_h.numel() * 2

    cpu = None
    if keep_inputs:
        t_cpu, rows_done = _cpu_baseline(cfg, dict(inp, **canon))
        cpu = {"value": ubytes / t_cpu / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "%d of %d rows of the same workload through the oracle, scaled to the full step"
                         % (rows_done, M)}

    if rank == 0:
        line = {"metric": METRIC, "value": gbs * world, "unit": "GB/s", "n_gpus": world, "steps": a.steps,
                "warmup": a.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": synth.FMT_NAMES[cfg["w_fmt"]],
                "data": "synthetic (seeded): inputs of the workload's shapes, random weights",
                "config": {"workload": cfg["name"], "rows": M, "H": H, "E": cfg["E"], "k": cfg["k"], "I": I,
                           "shared_I": Ish, "swiglu_limit": cfg.get("swiglu_limit", 0.0),
                           "unique_experts": n_active, "unique_bytes": ubytes,
                           "us_per_step": ms_step * 1e3, "rows_per_s": M / (ms_step * 1e-3),
                           "frac_of_measured_peak": gbs / peak, "frac_of_8000": gbs / 8000.0,
                           "l2": "512 MiB buffer written, then another 512 MiB read, between timed steps (untimed)",
                           "parallelism": "replicas" if world > 1 else "single GPU",
                           "wall_s_timed_region": wall},
                "e2e": {"value": ubytes / e2e_s / 1e9 * world, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3},
                "roofline": roofline, "cpu_baseline": cpu, "clocks": clk,
                "gpu_launches": (4 if fused else 5) * a.steps}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
