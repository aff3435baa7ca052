"""The bench's multi-process path on CPU (gloo, world size 2): the whole-job
reductions and the reference arm under torchrun.  The GPU arm's replicas use
the same reductions; the layer itself has no exchange step (replicas only)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    import synth as S
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slow = bench.reduce_ranks(10.0 + 5.0 * rank, world, "max")
        count = bench.reduce_ranks(3.0 + rank, world, "sum")
        wl = bench.replica_workload(S.WORKLOADS["tiny_w8a16"], rank)
        q.put((rank, slow, count, wl.seed))
    finally:
        dist.destroy_process_group()


def test_reductions_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    # both ranks see the slowest replica's time and the summed count
    assert [g[1] for g in got] == [15.0, 15.0]
    assert [g[2] for g in got] == [7.0, 7.0]
    # replicas draw independent batches
    assert got[0][3] != got[1][3]


def test_reduction_is_identity_at_one_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_ranks(12.5, 1, "max") == 12.5
    assert bench.reduce_ranks(4.0, 1, "sum") == 4.0


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_prints_one_line_from_rank0():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--workload", "tiny_w8a16", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=280)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_gate_up_algorithmic_bytes_by_hand():
    """The roofline numerator, counted independently from the formats' storage
    rules: per touched expert the gate and up codes and scales, plus the
    gathered activation rows read and h written once."""
    sys.path.insert(0, ROOT)
    import bench
    import synth as S
    wl = S.WORKLOADS["decode_w4a16"]      # INT4: 0.5 B/code, FP16 scale per 128
    P, H, I = wl.T * wl.k, wl.H, wl.I
    per_expert = 2 * (I * H // 2 + I * (H // 128) * 2)
    assert bench.gate_up_bytes(wl, 256) == 256 * per_expert + P * H * 2 + P * I * 2 == 287309824
    wl = S.WORKLOADS["w8a8_2048"]         # INT8 codes, INT8 activations with an FP32 scale per 128
    P, H, I = wl.T * wl.k, wl.H, wl.I
    per_expert = 2 * (I * H + I * (H // 128) * 2)
    assert bench.gate_up_bytes(wl, 256) == 256 * per_expert + P * (H + H // 128 * 4) + P * I * 2
    wl = S.WORKLOADS["prefill_nvfp4"]     # E2M1 codes, E4M3 per 16, FP32 outer per matrix; same for activations
    P, H, I = wl.T * wl.k, wl.H, wl.I
    per_expert = 2 * (I * H // 2 + I * (H // 16) + 4)
    assert bench.gate_up_bytes(wl, 200) == 200 * per_expert + P * (H // 2 + H // 16 + 4) + P * I * 2


def test_gpu_arm_json_line_contract():
    """The GPU arm's JSON line, built from fabricated measurements: every key of
    the contract, the whole-job value, and the roofline bound chosen by
    arithmetic intensity (HBM for the decode batch, tensor for the large
    W4A16 batch)."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    import synth as S
    args = argparse.Namespace(steps=10, warmup=3)
    hbm, bf16, kind = bench._peaks()
    for name, step_ms, gu_ms, bound in (("decode_w4a16", 0.1351, 0.0785, "hbm"),
                                        ("large_w4a16", 1.9172, 1.1123, "tensor")):
        wl = S.WORKLOADS[name]
        ids = S.routing_uniform(wl.T, wl.E, wl.k, seed=1)
        r = dict(total_ms=10 * step_ms, step_ms=[step_ms] * 10, gu_ms=[gu_ms] * 10, touched=wl.E, ids=ids,
                 e2e_ms=0.174, world=2, launches=100, f16_rows=True,
                 clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []})
        line = bench.build_line(args, wl, {"workload": name}, r, (4.4, 10.0, 12), (12345, "test"))
        for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                    "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                    "gpu_launches", "clocks"):
            assert key in line, key
        assert line["value"] == pytest.approx(2 * wl.T / (step_ms / 1e3))  # whole job: both replicas
        assert line["n_gpus"] == 2 and line["scaling"] == "weak" and line["higher_is_better"] is True
        roof = line["roofline"]
        for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
            assert key in roof, key
        assert roof["bound"] == bound and roof["traffic"] == 12345
        assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
        if bound == "hbm":
            assert roof["peak"] == hbm and roof["unit"] == "GB/s"
            assert roof["achieved"] == pytest.approx(bench.gate_up_bytes(wl, wl.E) / (gu_ms / 1e3) / 1e9)
        else:
            assert roof["peak"] == bf16 and roof["unit"] == "TFLOP/s"
            assert roof["achieved"] == pytest.approx(2 * 2 * wl.H * wl.I * wl.T * wl.k / (gu_ms / 1e3) / 1e12)
        assert roof["launch_ms_median"] == pytest.approx(gu_ms)
        assert line["ms_per_step_median"] == pytest.approx(step_ms)
        assert line["dtype"].startswith("f16 x f16")  # INT4 weights on FP16 rows
        cb = line["cpu_baseline"]
        assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == 4.4 and "sample" in cb
        assert cb["host_nproc"] == os.cpu_count() and cb["host_cpu_model"]
        e2e = line["e2e"]
        assert e2e["value"] == pytest.approx(2 * wl.T / 0.174e-3)
        assert e2e["h2d_bytes_per_step"] == 2 * (wl.T * wl.H * 2 + wl.T * wl.k * 8)
        assert e2e["d2h_bytes_per_step"] == 2 * wl.T * wl.H * 2
        assert "variants" not in line and "graph" not in line  # only when measured
    # the comparison paths and the graph replay pass through with their notes
    r.update(variants={"routed_forward_ms": 0.15, "route_ms": 0.02, "host_routing_forward_ms": 0.74,
                       "unfused_forward_ms": 0.17, "fused_forward_ms": 0.135}, graph_ms=0.134)
    line = bench.build_line(args, wl, {"workload": name}, r, (4.4, 10.0, 12), (12345, "test"))
    assert line["variants"]["route_ms"] == 0.02 and "note" in line["variants"]
    assert line["graph"]["ms_per_step_median"] == 0.134
    assert line["graph"]["value"] == pytest.approx(2 * wl.T / 0.134e-3)
    # the captured traffic is read from the committed ncu summary table, and
    # reported only while the GEMM sources hash to the value recorded with it
    table = os.path.join(ROOT, "profiles", "gate_up_dram_traffic.txt")
    for ln in open(table):
        parts = ln.split()
        if parts and not ln.startswith("#"):
            got, note = bench.profile_traffic(S.WORKLOADS[parts[0]])
            if parts[2] == bench.gemm_source_hash():
                assert got == int(parts[1])
            else:
                assert got is None and note.startswith("stale")
    assert bench.profile_traffic(S.WORKLOADS["tiny_w8a16"])[0] is None


def test_fp4_tensor_peak_is_measured_or_nominal():
    """NVFP4 fractions are quoted against an FP4 peak: the measured figure when
    profiles/tensor_peaks_gb300.json exists, else BF16 x the nominal 6."""
    sys.path.insert(0, ROOT)
    import bench
    hbm, bf16, kind = bench._peaks()
    peak, how = bench.tensor_peak("fp4", bf16, kind)
    if os.path.exists(os.path.join(ROOT, "profiles", "tensor_peaks_gb300.json")):
        assert how.startswith("measured") and peak > bf16
    else:
        assert peak == pytest.approx(6 * bf16) and "nominal" in how
    assert bench.tensor_peak("f16", bf16, kind)[0] == bf16


def test_attention_flop_count_matches_brute_force():
    import bench
    import synth as S
    aw = S.AttnWorkload("t", 2, 70, 3, 1, 16, 32, 0)
    allowed = sum(1 for t in range(aw.T) for j in range(aw.T) if j // aw.blk <= t // aw.blk)
    assert bench.attn_flops(aw) == 4.0 * aw.d * aw.Hq * aw.B * allowed
    assert 1 <= bench.attn_cpu_rows(aw, 1e-9) <= aw.B * aw.T
    assert bench.attn_cpu_rows(aw, 1e9) == aw.B * aw.T
