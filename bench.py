"""Benchmark of the routed-expert MoE layer on GB300.

One step = one pass of the whole layer (permute + gather, fused gate/up/SiLU
grouped GEMM, down grouped GEMM, combine; plus the activation quantisers in
the A8/A4 modes) over one batch of seeded synthetic inputs already resident in
HBM.  The default workload is the largest single-GPU one: 4096 tokens,
H=4096, 256 experts, I=1536, top-8, INT4 weights with FP16 scales per 128
(W4A16), skewed routing.  --workload picks another.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores instead (a bounded sample of the same workload).  --peaks runs the
tensor-core peak microbenchmark (bench_peaks.cu) and prints its JSON.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth as S  # noqa: E402

METRIC = "MoE-layer tokens/s and achieved HBM GB/s or tensor-pipe % vs GB300 peak, 1 GPU"
ATTN_METRIC = "Block-attention prefill tokens/s and achieved tensor-pipe % vs GB300 peak, 1 GPU"
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# Dense tensor rates relative to BF16 on GB300 (nominal: 2.25 PFLOP/s BF16/FP16,
# 13.5 FP4).  Used only where no measured figure of that MMA kind exists.
NOMINAL_RATIO = {"bf16": 1.0, "f16": 1.0, "fp4": 6.0}


def tensor_peak(mma: str, bf16_peak: float, bf16_kind: str):
    """Peak (TFLOP/s) of the MMA kind a gate/up launch issues, and how it was
    obtained.  BF16 and FP16: the measured cuBLAS BF16 burst peak (FP16 runs
    at the BF16 rate).  FP4: the figure profiles/tensor_peaks_gb300.json holds
    (written by `python bench.py --peaks` on a GB300) when present, else the
    measured BF16 peak times the nominal FP4/BF16 ratio."""
    if mma in ("bf16", "f16"):
        return bf16_peak, f"{bf16_kind} (bf16 dense burst; f16 runs at the bf16 rate)"
    try:
        with open(os.path.join(ROOT, "profiles", "tensor_peaks_gb300.json")) as f:
            return float(json.load(f)["mxf4nvf4_tflops"]), "measured (tcgen05 microbenchmark, bench_peaks.cu)"
    except (OSError, KeyError, ValueError):
        return bf16_peak * NOMINAL_RATIO[mma], f"{bf16_kind} bf16 x nominal {NOMINAL_RATIO[mma]:g}"


def run_peaks() -> dict:
    """Build bench_peaks.cu with nvcc and run it on the current GPU; returns its
    JSON (dense TFLOP/s of tcgen05 kind::f16 and kind::mxf4nvf4)."""
    exe = os.path.join("/tmp", f"bench_peaks_{os.getpid()}")
    nvcc = os.environ.get("NVCC", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-o", exe,
                    os.path.join(ROOT, "bench_peaks.cu")], check=True)
    try:
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=300).stdout
    finally:
        os.remove(exe)
    return json.loads(out.strip().splitlines()[-1])


def host_info():
    """nproc and CPU model of the host this process runs on."""
    model = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = ln.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model in ("", "aarch64"):
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
            for ln in out.splitlines():
                if ln.lower().startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return os.cpu_count(), model


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_ranks(value: float, world: int, op: str, device=None) -> float:
    """Whole-job value of a per-rank number: "max" (times: the slowest replica
    sets the job's time) or "sum" (counts).  World size 1 returns the value."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX if op == "max" else torch.distributed.ReduceOp.SUM)
    return float(t.item())


def replica_workload(wl: S.Workload, rank: int) -> S.Workload:
    """Replicas run independent batches: rank r draws its inputs from seed + 1000 r."""
    return dataclasses.replace(wl, seed=wl.seed + 1000 * rank) if rank else wl


def gate_up_bytes(wl: S.Workload, touched: int) -> int:
    """Algorithmic bytes of one gate/up launch: each touched expert's gate and up
    matrices (codes + scales) once, the gathered activations read once, h written once."""
    L = S.layout(wl.wfmt, wl.E, wl.H, wl.I)
    per_expert = 0
    for m in (S.GATE, S.UP):
        N, K = L.dims(m)
        per_expert += S.code_bytes(wl.wfmt, N, K) + S.scale_bytes(wl.wfmt, N, K)
        per_expert += 4 if wl.wfmt == S.FMT_NVFP4_G16 else 0  # the matrix's FP32 outer scale
    act = {S.ACT_BF16: wl.H * 2, S.ACT_INT8_G128: wl.H + wl.H // 128 * 4,
           S.ACT_NVFP4_G16: wl.H // 2 + wl.H // 16 + 4}[wl.act]
    return touched * per_expert + wl.P * act + wl.P * wl.I * 2


def run_ours(args, wl):
    import quantized_moe_expert_routed_gb300 as M

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    x, ids, w, blob, hdr, L = S.make_inputs(replica_workload(wl, rank), device=dev)
    layer = M.Layer(blob, hdr)
    M.mnw_moe_set_gemm_path({"auto": M.PATH_AUTO, "tcgen05": M.PATH_TCGEN05, "warp": M.PATH_WARP_MMA,
                             "rows": M.PATH_ROWS}[args.gemm_path])
    E, T, k, P = wl.E, wl.T, wl.k, wl.P
    stream = torch.cuda.current_stream(dev)
    ws = M.workspace(layer, wl.act, T, k, device=dev)
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    flush_clean = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def l2_flush():
        # Write a buffer larger than L2, then read another one: the dirty lines
        # the write leaves behind are written back here, not inside the next
        # timed kernel, which starts with an L2 holding none of its inputs.
        flush.zero_()
        flush_clean.amax()

    # Preallocated per-step buffers for the stepwise path (same kernels as mnw_moe_forward,
    # called one by one so the gate/up launch can be timed on its own stream).
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_assign = torch.empty(P, dtype=torch.int32, device=dev)
    assign_pos = torch.empty(P, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib = M.load()
    import ctypes
    sp = ctypes.c_void_p(stream.cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    gemm_name = {(S.FMT_BF16, S.ACT_BF16): "bf16", (S.FMT_INT8_G128, S.ACT_BF16): "w8a16",
                 (S.FMT_INT4_G128, S.ACT_BF16): "w4a16", (S.FMT_INT8_G128, S.ACT_INT8_G128): "w8a8",
                 (S.FMT_INT4_G128, S.ACT_INT8_G128): "w4a8",
                 (S.FMT_NVFP4_G16, S.ACT_NVFP4_G16): "nvfp4"}[(wl.wfmt, wl.act)]
    gemm = getattr(lib, f"mnw_moe_grouped_gemm_{gemm_name}")
    h = torch.empty((P, wl.I), dtype=torch.bfloat16, device=dev)
    y = torch.empty((P, wl.H), dtype=torch.bfloat16, device=dev)
    if wl.act == S.ACT_BF16:
        xa = torch.empty((P, wl.H), dtype=torch.bfloat16, device=dev)
    elif wl.act == S.ACT_INT8_G128:
        xq = torch.empty((P, wl.H), dtype=torch.int8, device=dev)
        xs = torch.empty((P, wl.H // 128), dtype=torch.float32, device=dev)
        hq = torch.empty((P, wl.I), dtype=torch.int8, device=dev)
        hs = torch.empty((P, wl.I // 128), dtype=torch.float32, device=dev)
    else:
        xq = torch.empty((P, wl.H // 2), dtype=torch.uint8, device=dev)
        xs = torch.empty((P, wl.H // 16), dtype=torch.uint8, device=dev)
        xo = torch.empty((P,), dtype=torch.float32, device=dev)
        hq = torch.empty((P, wl.I // 2), dtype=torch.uint8, device=dev)
        hs = torch.empty((P, wl.I // 16), dtype=torch.uint8, device=dev)
        ho = torch.empty((P,), dtype=torch.float32, device=dev)

    def chk(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} failed: {lib.mnw_status_string(rc).decode()}")

    # INT weights with BF16 activations: the forward runs gate/up on FP16 rows
    # (row factor in xf), and down too once there are enough tokens per expert
    # for the tcgen05 kernel, so the stepwise sequence and the roofline loop
    # do the same.
    f16_gate_up = f16_down = None
    if wl.act == S.ACT_BF16 and wl.wfmt in (S.FMT_INT8_G128, S.FMT_INT4_G128):
        f16 = getattr(lib, f"mnw_moe_grouped_gemm_{gemm_name}_f16rows")
        # a zero-row call reports whether the layer's scales allow the FP16 form
        allowed = [f16(layer.handle, kind, None, None, None, 0, None, None, sp) == 0 for kind in (0, 1)]
        allowed[1] = allowed[1] and (-(-P // E) >= 32 or args.gemm_path in ("tcgen05", "rows"))
        if allowed[0]:
            f16_gate_up = f16
            xa = torch.empty((P, wl.H), dtype=torch.float16, device=dev)
            xf = torch.empty((P,), dtype=torch.float32, device=dev)
        if allowed[1]:
            f16_down = f16
            ha = torch.empty((P, wl.I), dtype=torch.float16, device=dev)
            hf = torch.empty((P,), dtype=torch.float32, device=dev)

    def step():
        """The layer's kernels called one by one (prepares the gate/up inputs)."""
        if wl.act == S.ACT_BF16:
            if f16_gate_up is not None:
                chk(lib.mnw_moe_permute(ptr(ids), T, k, E, ptr(offsets), ptr(sorted_assign), ptr(assign_pos), None,
                                        0, None, ptr(err), sp), "permute")
                chk(lib.mnw_moe_quantize_act(M.ACT_F16_ROWS, ptr(x), P, wl.H, ptr(sorted_assign), k, ptr(xa), None,
                                             ptr(xf), sp), "encode x")
                chk(f16_gate_up(layer.handle, 0, ptr(xa), ptr(xf), ptr(offsets), P, ptr(h), ptr(err), sp), "gate_up")
            else:
                chk(lib.mnw_moe_permute(ptr(ids), T, k, E, ptr(offsets), ptr(sorted_assign), ptr(assign_pos), ptr(x),
                                        wl.H, ptr(xa), ptr(err), sp), "permute")
                chk(gemm(layer.handle, 0, ptr(xa), ptr(offsets), P, ptr(h), ptr(err), sp), "gate_up")
            if f16_down is not None:
                chk(lib.mnw_moe_quantize_act(M.ACT_F16_ROWS, ptr(h), P, wl.I, None, 1, ptr(ha), None, ptr(hf), sp),
                    "encode h")
                chk(f16_down(layer.handle, 1, ptr(ha), ptr(hf), ptr(offsets), P, ptr(y), ptr(err), sp), "down")
            else:
                chk(gemm(layer.handle, 1, ptr(h), ptr(offsets), P, ptr(y), ptr(err), sp), "down")
        else:
            chk(lib.mnw_moe_permute(ptr(ids), T, k, E, ptr(offsets), ptr(sorted_assign), ptr(assign_pos), None, 0,
                                    None, ptr(err), sp), "permute")
            o1 = ptr(xo) if wl.act == S.ACT_NVFP4_G16 else None
            o2 = ptr(ho) if wl.act == S.ACT_NVFP4_G16 else None
            chk(lib.mnw_moe_quantize_act(wl.act, ptr(x), P, wl.H, ptr(sorted_assign), k, ptr(xq), ptr(xs), o1, sp),
                "quantize x")
            if wl.act == S.ACT_INT8_G128:
                chk(gemm(layer.handle, 0, ptr(xq), ptr(xs), ptr(offsets), P, ptr(h), None, ptr(err), sp), "gate_up")
            else:
                chk(gemm(layer.handle, 0, ptr(xq), ptr(xs), o1, ptr(offsets), P, ptr(h), ptr(err), sp), "gate_up")
            chk(lib.mnw_moe_quantize_act(wl.act, ptr(h), P, wl.I, None, 1, ptr(hq), ptr(hs), o2, sp), "quantize h")
            if wl.act == S.ACT_INT8_G128:
                chk(gemm(layer.handle, 1, ptr(hq), ptr(hs), ptr(offsets), P, ptr(y), None, ptr(err), sp), "down")
            else:
                chk(gemm(layer.handle, 1, ptr(hq), ptr(hs), o2, ptr(offsets), P, ptr(y), ptr(err), sp), "down")
        chk(lib.mnw_moe_combine(ptr(y), ptr(assign_pos), ptr(w), T, k, wl.H, ptr(out), sp), "combine")

    # Headline: whole layer steps through the library's one-call entry point
    # (its kernels launch back to back with programmatic dependent launch; no
    # event sits between them).
    ws_bytes = ws.numel()
    fwd = lib.mnw_moe_forward

    def layer_step():
        chk(fwd(layer.handle, wl.act, ptr(x), ptr(ids), ptr(w), T, k, ptr(out), ptr(ws), ws_bytes, sp), "forward")

    def gate_up_only():
        if f16_gate_up is not None:
            chk(f16_gate_up(layer.handle, 0, ptr(xa), ptr(xf), ptr(offsets), P, ptr(h), ptr(err), sp), "gate_up")
        elif wl.act == S.ACT_BF16:
            chk(gemm(layer.handle, 0, ptr(xa), ptr(offsets), P, ptr(h), ptr(err), sp), "gate_up")
        elif wl.act == S.ACT_INT8_G128:
            chk(gemm(layer.handle, 0, ptr(xq), ptr(xs), ptr(offsets), P, ptr(h), None, ptr(err), sp), "gate_up")
        else:
            chk(gemm(layer.handle, 0, ptr(xq), ptr(xs), ptr(xo), ptr(offsets), P, ptr(h), ptr(err), sp), "gate_up")

    for _ in range(args.warmup):
        layer_step()
        l2_flush()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    launches = 0
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            l2_flush()  # between timed iterations, outside the events
            e0, e1 = ev[i]
            e0.record(stream)
            n0 = lib.mnw_moe_launch_count()
            layer_step()
            launches += lib.mnw_moe_launch_count() - n0  # the library's own kernels, counted by the library
            e1.record(stream)
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = reduce_ranks(sum(step_ms), world, "max", dev)
    launches = int(reduce_ranks(launches, world, "sum", dev))
    e = M.mnw_moe_read_error(M.workspace_error_word(ws))
    if e:
        raise RuntimeError(f"device error word {e:#x}")

    # The same forward captured once in a CUDA graph and replayed: the host's
    # launch work leaves the step (the kernels and their order are unchanged).
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap):
        chk(fwd(layer.handle, wl.act, ptr(x), ptr(ids), ptr(w), T, k, ptr(out), ptr(ws), ws_bytes,
                ctypes.c_void_p(cap.cuda_stream)), "forward (graph capture)")
    stream.wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize()
    gr_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        l2_flush()
        a0, a1 = gr_ev[i]
        a0.record(stream)
        graph.replay()
        a1.record(stream)
    torch.cuda.synchronize()
    graph_ms = reduce_ranks(statistics.median([a.elapsed_time(b) for a, b in gr_ev]), world, "max", dev)
    e = M.mnw_moe_read_error(M.workspace_error_word(ws))
    if e:
        raise RuntimeError(f"device error word {e:#x} after graph replays")
    del graph

    # Roofline: the fused gate/up GEMM launch alone, on inputs prepared by the
    # same kernels as the layer (CUDA events on its stream, L2 flushed between).
    step()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps + 1):
        l2_flush()
        if i == 0:
            gate_up_only()  # warm
            continue
        g0, g1 = gev[i - 1]
        g0.record(stream)
        gate_up_only()
        g1.record(stream)
    torch.cuda.synchronize()
    gu_ms = [a.elapsed_time(b) for a, b in gev]
    if int(err.item()):
        raise RuntimeError(f"device error word {int(err.item()):#x}")

    # end-to-end through the host-buffer entry point (copies inside the timed region)
    wsh = M.workspace(layer, wl.act, T, k, host=True, device=dev)
    xh, idh, wh = x.cpu().pin_memory(), ids.cpu().pin_memory(), w.cpu().pin_memory()
    outh = torch.empty((T, wl.H), dtype=torch.bfloat16).pin_memory()
    for _ in range(max(1, args.warmup)):
        M.mnw_moe_forward_host(layer, wl.act, xh, idh, wh, wsh, outh)
    e2e_ms = []
    for _ in range(args.steps):
        l2_flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        M.mnw_moe_forward_host(layer, wl.act, xh, idh, wh, wsh, outh)
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_ms = reduce_ranks(statistics.median(e2e_ms), world, "max", dev)

    # The comparison paths the pages describe, on the same input (device buffers,
    # L2 flushed between steps, CUDA events, median): GPU routing fused with the
    # permutation (router weights ~N(0, 1/H) in BF16), the router alone, the
    # unfused activation, and host routing (it synchronises: wall clock).
    variants = {}
    nv = max(3, min(args.steps, 10))

    def timed(fn, wall=False):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(nv):
            l2_flush()
            if wall:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                fn()
                torch.cuda.synchronize()
                ts.append((time.perf_counter() - t0) * 1e3)
            else:
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                fn()
                a1.record(stream)
                torch.cuda.synchronize()
                ts.append(a0.elapsed_time(a1))
        return statistics.median(ts)

    try:
        wr = S.router_weights(E, wl.H, wl.seed, device=dev)
        wsr = torch.empty(M.mnw_moe_workspace_size_routed(layer, wl.act, T, k) + 256, dtype=torch.uint8, device=dev)
        outr = torch.empty_like(out)
        scratch = torch.zeros(lib.mnw_moe_route_scratch_size(T, E) + 256, dtype=torch.uint8, device=dev)
        routed = lambda: M.mnw_moe_forward_routed(layer, wl.act, x, wr, k, ws=wsr, out=outr)  # noqa: E731
        variants["routed_forward_ms"] = timed(routed)
        r_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        r_w = torch.empty((T, k), dtype=torch.float32, device=dev)
        r_off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        r_sa = torch.empty(P, dtype=torch.int32, device=dev)
        r_pos = torch.empty(P, dtype=torch.int32, device=dev)
        r_base = (-scratch.data_ptr()) % 256
        r_need = lib.mnw_moe_route_scratch_size(T, E)

        def route():
            chk(lib.mnw_moe_route(ptr(x), ptr(wr), T, wl.H, E, k, ptr(r_ids), ptr(r_w), ptr(r_off), ptr(r_sa),
                                  ptr(r_pos), ctypes.c_void_p(scratch.data_ptr() + r_base), r_need, ptr(err), sp),
                "route")

        variants["route_ms"] = timed(route)
        M.mnw_moe_set_host_routing(True)
        try:
            variants["host_routing_forward_ms"] = timed(routed, wall=True)
        finally:
            M.mnw_moe_set_host_routing(False)
    except Exception as ex:  # a shape the router does not take
        variants["routed_note"] = f"not timed: {ex}"
    M.mnw_moe_set_fused_activation(False)
    try:
        variants["unfused_forward_ms"] = timed(layer_step)
    finally:
        M.mnw_moe_set_fused_activation(True)
    variants["fused_forward_ms"] = timed(layer_step)

    touched = int(torch.unique(ids[(ids >= 0) & (ids < E)]).numel())
    return dict(total_ms=total_ms, step_ms=step_ms, gu_ms=gu_ms, launches=launches, world=world, rank=rank,
                f16_rows=f16_gate_up is not None, graph_ms=graph_ms, variants=variants,
                clocks=clk.summary(), e2e_ms=e2e_ms, touched=touched, ids=ids)


def cpu_sample_tokens(wl: S.Workload, budget_s: float):
    """How many tokens of the workload the oracle runs in about budget_s seconds."""
    macs_per_token = 3 * wl.H * wl.I * wl.k
    rate = 6.0e7 if wl.wfmt != S.FMT_BF16 else 1.0e8  # oracle MAC/s (single thread, with decode)
    return max(1, min(wl.T, int(budget_s * rate / macs_per_token)))


def run_oracle_sample(wl: S.Workload, ntok: int, inputs=None):
    import oracle
    if inputs is None:
        x, ids, w, blob, hdr, L = S.make_inputs(wl, device="cuda" if torch.cuda.is_available() else "cpu")
    else:
        x, ids, w, blob = inputs
    rows = np.linspace(0, wl.T - 1, ntok).astype(np.int32)
    b = blob.cpu().numpy()
    xb, idn, wn = S.bf16_bits_np(x), ids.cpu().numpy(), w.cpu().numpy()
    t0 = time.perf_counter()
    oracle.moe_forward(b, wl.act, xb, idn, wn, rows=rows)
    dt = time.perf_counter() - t0
    return ntok / dt, dt


GEMM_SOURCES = ("mnw_gemm", "mnw_convert.cuh", "mnw_ptx.cuh")


def gemm_source_hash(prefixes=None) -> str:
    """First 12 hex digits of a SHA-256 over the grouped-GEMM kernel sources
    (every csrc file whose name starts with one of GEMM_SOURCES, or of the
    prefixes given), in name order."""
    csrc = os.path.join(ROOT, "quantized_moe_expert_routed_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.startswith(prefixes or GEMM_SOURCES):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:12]


ATTN_SOURCES = ("mnw_attention", "mnw_convert.cuh", "mnw_ptx.cuh")


def profile_traffic(wl, table="gate_up_dram_traffic.txt", sources=None):
    """DRAM traffic (read + write bytes) of one launch of the dominant kernel,
    from the ncu capture summarised in profiles/ (lines "<workload> <bytes>
    <source hash> <summary file>"), and a note.  The figure is None when there
    is no line for the workload, or when the kernel sources changed since the
    capture (their hash differs from the one recorded beside it)."""
    try:
        with open(os.path.join(ROOT, "profiles", table)) as f:
            for ln in f:
                parts = ln.split()
                if len(parts) >= 3 and parts[0] == wl.name:
                    now = gemm_source_hash(sources)
                    if parts[2] != now:
                        sys.stderr.write(f"bench: stored DRAM traffic for {wl.name} predates the current kernel "
                                         f"sources ({parts[2]} != {now}); reporting null\n")
                        return None, "stale: the kernel changed since the capture"
                    return int(parts[1]), f"ncu capture, profiles/{parts[3] if len(parts) > 3 else ''}"
    except OSError:
        pass
    return None, "no capture of the current kernel"


def gate_up_mma(wl: S.Workload, f16_rows: bool) -> tuple:
    """(MMA kind the gate/up launch issues, dtype string of the path)."""
    if wl.act == S.ACT_NVFP4_G16:
        return "fp4", "e2m1 x e2m1, e4m3 block scales, fp32 outer scales -> f32 (block-scaled fp4 MMA)"
    if wl.act == S.ACT_INT8_G128:
        return "f16", "int8 x int8 group dots exact in f16 MMA (f32 accumulate) -> f32 group combine"
    if wl.wfmt == S.FMT_BF16:
        return "bf16", "bf16 x bf16 -> f32"
    w = "int4" if wl.wfmt == S.FMT_INT4_G128 else "int8"
    if f16_rows:
        return "f16", (f"f16 x f16 -> f32 ({w} weights dequantised on chip; bf16 rows re-encoded exactly as f16 "
                       "with a power-of-two row factor)")
    return "bf16", f"bf16 x bf16 -> f32 ({w} codes as exact bf16 integers, f32 group scales)"


def build_line(args, wl: S.Workload, config: dict, r: dict, cpu, traffic) -> dict:
    """The JSON line of the GPU arm from run_ours' measurements r, the CPU
    baseline (tokens/s, seconds, sample tokens) and the captured traffic
    (bytes or None, note)."""
    hbm, bf16_peak, peak_kind = _peaks()
    ms = r["total_ms"] / args.steps
    value = r["world"] * wl.T / (r["total_ms"] / args.steps / 1e3)
    gu_ms = statistics.mean(r["gu_ms"])
    gu_bytes = gate_up_bytes(wl, r["touched"])
    achieved = gu_bytes / (gu_ms / 1e3) / 1e9
    # The gate/up launch's binding roofline: its arithmetic intensity against
    # the ridge of the HBM peak and the dense peak of the MMA kind it issues
    # (the kernel is timed alone: the burst figure).
    mma, dtype = gate_up_mma(wl, r.get("f16_rows", False))
    t_peak, t_kind = tensor_peak(mma, bf16_peak, peak_kind)
    valid = int(((r["ids"] >= 0) & (r["ids"] < wl.E)).sum())
    gu_flops = 2.0 * 2 * wl.H * wl.I * valid
    gu_tflops = gu_flops / (gu_ms / 1e3) / 1e12
    tensor_bound = gu_flops / gu_bytes > t_peak * 1e12 / (hbm * 1e9)
    layer_bytes = S.algorithmic_bytes(wl, r["ids"].cpu())
    e2e_ms = r["e2e_ms"]  # the slowest replica's median
    h2d = r["world"] * (wl.T * wl.H * 2 + wl.P * 4 * 2)  # x, ids, w of every replica
    d2h = r["world"] * wl.T * wl.H * 2
    cpu_rate, cpu_dt, ntok = cpu
    nproc, cpu_model = host_info()
    traffic_bytes, traffic_note = traffic
    tensor = {"achieved": gu_tflops, "peak": t_peak, "unit": "TFLOP/s", "frac": gu_tflops / t_peak,
              "peak_kind": t_kind, "mma": mma, "flops_per_launch": gu_flops}
    hbm_part = {"achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "peak_kind": peak_kind,
                "bytes_per_launch": gu_bytes}
    if tensor_bound:
        roofline = {"kernel": "grouped gate/up/SiLU GEMM", "bound": "tensor", **tensor, "launch_ms": gu_ms,
                    "launch_ms_median": statistics.median(r["gu_ms"]), "traffic": traffic_bytes,
                    "traffic_note": traffic_note, "hbm": hbm_part}
    else:
        roofline = {"kernel": "grouped gate/up/SiLU GEMM", "bound": "hbm", **hbm_part, "launch_ms": gu_ms,
                    "launch_ms_median": statistics.median(r["gu_ms"]), "traffic": traffic_bytes,
                    "traffic_note": traffic_note, "tensor": tensor}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": r["world"], "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": statistics.median(r["step_ms"]),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic (seeded, shapes of the workload)",
        "config": config,
        "layer_effective_gbs": layer_bytes / (ms / 1e3) / 1e9,
        "roofline": roofline,
        "cpu_baseline": {"value": cpu_rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "host_nproc": nproc, "host_cpu_model": cpu_model,
                         "sample": f"{ntok} of {wl.T} tokens, {cpu_dt:.1f} s single-threaded"},
        "e2e": {"value": r["world"] * wl.T / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if r.get("variants"):
        line["variants"] = {**r["variants"], "note": "comparison paths on the same batch, median ms per forward; "
                                                      "routed: the router's own expert choice (BF16 weights ~N(0, 1/H))"}
    if r.get("graph_ms"):
        line["graph"] = {"value": r["world"] * wl.T / (r["graph_ms"] / 1e3), "unit": "tokens/s",
                         "ms_per_step_median": r["graph_ms"],
                         "note": "the same forward captured once in a CUDA graph and replayed (L2 flushed between)"}
    return line


# ---------------------------------------------------------------------------
# the second workload: block attention for prompt prefill
# ---------------------------------------------------------------------------


def attn_flops(aw) -> float:
    """Useful FLOPs of one call: 2 products of 2*d flops per allowed (query, key)
    pair and query head (the masked pairs inside computed tiles not counted)."""
    t = np.arange(aw.T, dtype=np.int64)
    kend = np.minimum(aw.T, (t // aw.blk + 1) * aw.blk)
    return 4.0 * aw.d * aw.Hq * aw.B * float(kend.sum())


def attn_oracle_sample(aw, nrows: int, inputs):
    import oracle
    q, k, v = inputs
    rows = np.linspace(0, aw.B * aw.T - 1, nrows).astype(np.int32)
    u = lambda t: t.detach().cpu().contiguous().view(torch.uint16).numpy()  # noqa: E731
    qh, kh, vh = u(q), u(k), u(v)
    t0 = time.perf_counter()
    oracle.attention(qh, kh, vh, aw.blk, 1.0 / np.sqrt(aw.d), rows=rows)
    dt = time.perf_counter() - t0
    return nrows / dt, dt


def attn_cpu_rows(aw, budget_s: float) -> int:
    """How many query rows the oracle runs in about budget_s seconds (~4e8 FP64 MAC/s)."""
    macs_per_row = 2.0 * aw.Hq * aw.d * (aw.T / 2 + aw.blk)
    return max(1, min(aw.B * aw.T, int(budget_s * 4.0e8 / macs_per_row)))


def run_attn(args, aw):
    import ctypes

    import quantized_moe_expert_routed_gb300 as M
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank:
        aw = dataclasses.replace(aw, seed=aw.seed + 1000 * rank)
    q, k, v = S.attention_inputs(aw.B, aw.T, aw.Hq, aw.Hkv, aw.d, aw.seed, device=dev)
    lib = M.load()
    out = torch.empty_like(q)
    ws = torch.empty((lib.mnw_attn_workspace_size(aw.B, aw.T, aw.Hkv, aw.d),), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    scale = 1.0 / float(np.sqrt(aw.d))
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    flush_clean = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def l2_flush():
        flush.zero_()
        flush_clean.amax()

    def call(qq, kk, vv, oo):
        rc = lib.mnw_attn_prefill(ptr(qq), ptr(kk), ptr(vv), aw.B, aw.T, aw.Hq, aw.Hkv, aw.d, aw.blk,
                                  ctypes.c_float(scale), ptr(oo), ptr(ws), ws.numel(), ptr(err), sp)
        if rc != 0:
            raise RuntimeError(f"mnw_attn_prefill failed: {lib.mnw_status_string(rc).decode()}")

    for _ in range(args.warmup):
        call(q, k, v, out)
        l2_flush()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    launches = 0
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            l2_flush()
            e0, e1 = ev[i]
            e0.record(stream)
            n0 = lib.mnw_moe_launch_count()
            call(q, k, v, out)
            launches += lib.mnw_moe_launch_count() - n0
            e1.record(stream)
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = reduce_ranks(sum(step_ms), world, "max", dev)
    launches = int(reduce_ranks(launches, world, "sum", dev))
    if int(err.item()):
        raise RuntimeError(f"device error word {int(err.item()):#x}")

    # end to end: q, k, v from page-locked host memory, out back to it, inside the timed region
    qh, kh, vh = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    qd, kd, vd, od = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(out)

    def e2e_step():
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        call(qd, kd, vd, od)
        oh.copy_(od, non_blocking=True)
        stream.synchronize()

    for _ in range(max(1, args.warmup)):
        e2e_step()
    e2e_ms = []
    for _ in range(args.steps):
        l2_flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_ms = reduce_ranks(statistics.median(e2e_ms), world, "max", dev)
    return dict(total_ms=total_ms, step_ms=step_ms, launches=launches, world=world, rank=rank,
                clocks=clk.summary(), e2e_ms=e2e_ms, inputs=(q, k, v),
                h2d=q.numel() * 2 + k.numel() * 2 + v.numel() * 2, d2h=out.numel() * 2)


def attn_line(args, aw, r, cpu, traffic=(None, "no capture of the current kernel")) -> dict:
    hbm, bf16_peak, peak_kind = _peaks()
    ms = r["total_ms"] / args.steps
    flops = attn_flops(aw)
    achieved = flops / (ms / 1e3) / 1e12
    cpu_rate, cpu_dt, nrows = cpu
    nproc, cpu_model = host_info()
    tokens = aw.B * aw.T
    return {
        "metric": ATTN_METRIC, "value": r["world"] * tokens / (ms / 1e3), "unit": "tokens/s", "n_gpus": r["world"],
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "ms_per_step_median": statistics.median(r["step_ms"]), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 x bf16 -> f32 scores, f32 softmax, bf16 probabilities x bf16 -> f32",
        "data": "synthetic (seeded, shapes of the workload)",
        "config": {"workload": aw.name, "B": aw.B, "T": aw.T, "Hq": aw.Hq, "Hkv": aw.Hkv, "d": aw.d,
                   "mask": f"block-causal, {aw.blk}-token blocks",
                   "l2": "flushed between timed steps outside the events: a 2x L2 buffer written, then another "
                         "2x L2 buffer read"},
        "roofline": {"kernel": "block attention (the call: V transpose, then the attention kernel)",
                     "bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": achieved / bf16_peak, "peak_kind": f"{peak_kind} (bf16 dense burst)",
                     "flops_per_launch": flops, "launch_ms": ms, "launch_ms_median": statistics.median(r["step_ms"]),
                     "traffic": traffic[0], "traffic_note": traffic[1]},
        "cpu_baseline": {"value": cpu_rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "host_nproc": nproc, "host_cpu_model": cpu_model,
                         "sample": f"{nrows} of {tokens} query rows (all heads), {cpu_dt:.1f} s single-threaded"},
        "e2e": {"value": r["world"] * tokens / (r["e2e_ms"] / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": r["world"] * r["h2d"], "d2h_bytes_per_step": r["world"] * r["d2h"]},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }


def main_attn(args, aw):
    world, rank, local = _dist()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        if rank != 0:
            return
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        inputs = S.attention_inputs(aw.B, aw.T, aw.Hq, aw.Hkv, aw.d, aw.seed, device=dev)
        per_step = max(2.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
        nrows = attn_cpu_rows(aw, per_step)
        for _ in range(min(args.warmup, 1)):
            attn_oracle_sample(aw, max(1, nrows // 4), inputs)
        rates, times = [], []
        for _ in range(args.steps):
            rr, dt = attn_oracle_sample(aw, nrows, inputs)
            rates.append(rr)
            times.append(dt)
        value = statistics.median(rates)
        nproc, cpu_model = host_info()
        print(json.dumps({
            "impl": "reference", "metric": ATTN_METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(times) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": aw.name, "B": aw.B, "T": aw.T, "Hq": aw.Hq, "Hkv": aw.Hkv, "d": aw.d,
                       "mask": f"block-causal, {aw.blk}-token blocks"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "host_nproc": nproc,
                             "host_cpu_model": cpu_model,
                             "sample": f"{nrows} of {aw.B * aw.T} query rows per step (all heads)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return
    r = run_attn(args, aw)
    if rank != 0:
        return
    nrows = attn_cpu_rows(aw, args.cpu_budget)
    cpu = attn_oracle_sample(aw, nrows, r["inputs"])
    traffic = profile_traffic(aw, "attn_dram_traffic.txt", ATTN_SOURCES)
    print(json.dumps(attn_line(args, aw, r, (cpu[0], cpu[1], nrows), traffic)))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large_w4a16", choices=sorted(S.WORKLOADS) + sorted(S.ATTN_WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--peaks", action="store_true", help="run the tensor-core peak microbenchmark and exit")
    ap.add_argument("--gemm-path", default="auto", choices=["auto", "tcgen05", "warp", "rows"],
                    help="grouped-GEMM kernel selection (mnw_moe_set_gemm_path)")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's token count (smaller cases)")
    ap.add_argument("--experts", type=int, default=0, help="override the workload's expert count (smaller cases)")
    args = ap.parse_args()
    if args.peaks:
        print(json.dumps(run_peaks()))
        return
    if args.workload in S.ATTN_WORKLOADS:
        aw = S.ATTN_WORKLOADS[args.workload]
        if args.tokens:
            aw = dataclasses.replace(aw, name=f"{aw.name}_T{args.tokens}", T=args.tokens)
        main_attn(args, aw)
        return
    wl = S.WORKLOADS[args.workload]
    if args.tokens or args.experts:
        # a smaller case gets its own name, so no figure captured on the full workload is attached to it
        T_, E_ = args.tokens or wl.T, args.experts or wl.E
        wl = dataclasses.replace(wl, name=f"{wl.name}_T{T_}_E{E_}", T=T_, E=E_)
    world, rank, local = _dist()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    config = {"workload": wl.name, "T": wl.T, "H": wl.H, "E": wl.E, "I": wl.I, "k": wl.k, "gemm_path": args.gemm_path,
              "weights": ["bf16", "int8_g128", "int4_g128", "nvfp4_g16"][wl.wfmt],
              "activations": ["bf16", "int8_g128", "nvfp4_g16"][wl.act], "routing": wl.routing,
              "l2": "flushed between timed steps outside the events: a 2x L2 buffer written, then another 2x L2 buffer read"}

    if args.impl == "reference":
        if rank != 0:
            return
        per_step = max(2.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
        ntok = cpu_sample_tokens(wl, per_step)
        x, ids, w, blob, hdr, L = S.make_inputs(wl, device="cuda" if torch.cuda.is_available() else "cpu")
        inputs = (x, ids, w, blob)
        for _ in range(min(args.warmup, 1)):
            run_oracle_sample(wl, max(1, ntok // 4), inputs)
        rates, times = [], []
        for _ in range(args.steps):
            r, dt = run_oracle_sample(wl, ntok, inputs)
            rates.append(r)
            times.append(dt)
        value = statistics.median(rates)
        sample = f"{ntok} of {wl.T} tokens per step (token-by-token oracle, evenly spaced rows)"
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(times) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "host_nproc": host_info()[0], "host_cpu_model": host_info()[1], "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return

    r = run_ours(args, wl)
    if rank != 0:
        return
    # CPU baseline: the oracle on a bounded token sample, rank 0 only
    ntok = cpu_sample_tokens(wl, args.cpu_budget)
    cpu_rate, cpu_dt = run_oracle_sample(wl, ntok)
    line = build_line(args, wl, config, r, (cpu_rate, cpu_dt, ntok), profile_traffic(wl))
    print(json.dumps(line))


if __name__ == "__main__":
    main()
