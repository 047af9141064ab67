"""The multi-rank logic of bench.py on CPU: two gloo ranks, each with its own timing; the
job time is the slowest rank's and the job throughput counts every rank's tokens."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.max_over_ranks(10.0 + 3.5 * rank, "cpu")
    q.put((rank, slowest, bench.job_tokens_per_s(4096, world, 2.0)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in results] == [13.5, 13.5]
    assert all(abs(r[2] - 4096 * 2 / 0.002) < 1e-6 for r in results)


def test_single_process_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.0, "cpu") == 7.0
    assert bench.job_tokens_per_s(100, 1, 1.0) == 1e5


def test_reference_arm_json_line_on_cpu():
    """`bench.py --impl reference` runs the oracle on the host cores (no GPU) and prints
    one JSON line with the contract's keys, its cpu_baseline and e2e equal to its value."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_fp32", "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["config"]["workload"] == "tiny_fp32" and j["value"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] == j["value"]
    assert j["e2e"]["value"] == j["value"] and j["e2e"]["h2d_bytes_per_step"] == 0


def test_backward_floor_terms():
    """The backward's per-kernel roofline terms for the bf16_e64 shape, by hand: the
    weight-gradient kernels are HBM-bound by their fp32 outputs, the dx GEMM tensor-bound."""
    sys.path.insert(0, ROOT)
    import bench
    from synthetic import WORKLOADS
    w = WORKLOADS["bf16_e64"]
    pk = {"bf16_tflops": 1797.5, "hbm_gbs": 6484.3}
    N, d, f = 32768, 2048, 1024
    total, terms = bench.backward_floor(w, N, 64, pk)
    bw, tf = 6484.3e9, 1797.5e12
    assert abs(terms["wgrad_gate_up"] - (N * d * 2 + N * 2 * f * 2 + 64 * d * 2 * f * 4) / bw) < 1e-12
    assert abs(terms["wgrad_down"] - (N * f * 2 + N * d * 2 + 64 * f * d * 4) / bw) < 1e-12
    assert abs(terms["dx_gemm"] - 4.0 * N * d * f / tf) < 1e-12
    assert abs(total - sum(terms.values())) < 1e-15
    assert 650e-6 < total < 665e-6


def test_layer_bytes_and_flops():
    """The roofline numerators the bench reports, by hand: bf16_e64 (every expert local,
    N = T k) is tensor-bound in GEMM1 (4 N d f FLOP against 2 d f 2 B of weights per
    expert, the routed x rows and h); an EP64 MXFP8 slice counts E4M3 bytes plus one scale
    byte per 32 values, and only the non-empty experts' weights."""
    sys.path.insert(0, ROOT)
    import bench
    from synthetic import WORKLOADS
    w = WORKLOADS["bf16_e64"]
    T, d, f, E = 4096, 2048, 1024, 64
    N = T * 8
    b = bench.layer_bytes_flops(w, N, E, T)
    assert b["gemm1_flops"] == 4.0 * N * d * f and b["gemm2_flops"] == 2.0 * N * d * f
    assert b["layer_flops"] == b["gemm1_flops"] + b["gemm2_flops"]
    assert b["gemm1_bytes"] == 2 * d * f * 2 * E + N * d * 2 + N * f * 2
    assert b["gemm2_bytes"] == d * f * 2 * E + N * f * 2 + N * d * 2
    assert b["layer_bytes"] == 3 * d * f * 2 * E + T * d * 2 + T * d * 2 + T * E * 4
    # GEMM1 at bf16_e64: 275 GFLOP and 738 MB, tensor-bound against 1768 TFLOP/s and 6486 GB/s
    assert b["gemm1_flops"] / 1768.2e12 > b["gemm1_bytes"] / 6486.1e9
    m = WORKLOADS["mxfp8_ep64_T8192"]
    N, nonempty, tok = 1075, 4, 1000
    d, f = m.d, m.f
    b = bench.layer_bytes_flops(m, N, nonempty, tok)
    wb = pb = 1 + 1 / 32
    assert abs(b["gemm1_bytes"] - (2 * d * f * wb * nonempty + N * d * pb + N * f * pb)) < 1e-3
    assert abs(b["layer_bytes"] - (3 * d * f * wb * nonempty + tok * d * 2 + m.T * d * 2 + m.T * m.E * 4)) < 1e-3
    # the EP64 slice's GEMM1 is bound by its weight bytes
    assert b["gemm1_flops"] / 3536.4e12 < b["gemm1_bytes"] / 6486.1e9
