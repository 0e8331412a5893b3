"""Host-side logic of bench.py that needs no GPU: the algorithmic FLOP count
(visible pairs) against the oracle's brute-force count, and the multi-rank
timing reduction / input broadcast over world_size-2 gloo ranks, and the
reference arm (the oracle on the host cores) at one and two ranks."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads
from harness import problem_of

W = workloads.Workload


@pytest.mark.parametrize("w,lens", [
    (W("a", 2, 4, 2, 300, 300, 64, 64, causal=True), None),
    (W("b", 1, 2, 2, 200, 333, 64, 64, causal=True, bottom_right=True), None),
    (W("c", 1, 2, 2, 333, 200, 64, 64, causal=True, bottom_right=True), None),
    (W("d", 3, 2, 2, 300, 300, 64, 64, causal=True, window_left=64), np.array([1, 130, 300])),
    (W("e", 1, 2, 2, 260, 260, 64, 64, causal=True, window_right=50), None),
    (W("f", 1, 2, 2, 300, 280, 64, 64, window_left=150, bottom_right=True), None),
    (W("g", 2, 2, 2, 100, 100, 64, 64), np.array([0, 77])),
])
def test_visible_pairs_matches_oracle(oracle_mod, w, lens):
    p = problem_of(w, None if lens is None else torch.from_numpy(lens))
    assert bench.visible_pairs(w, lens) == oracle_mod.count_visible(p)


def test_headline_flops_formula():
    # D_qk = D_v = D: 2*(3D+2D) = 10*D per visible pair.
    w = workloads.WORKLOADS["causal_mha"]
    assert bench.flops_per_pair(w) == 10 * 128
    assert bench.visible_pairs(w, None) == 2 * 16 * 2048 * 2049 // 2


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    m = bench.max_over_ranks(1.5 + rank, world)
    t = torch.full((3,), float(rank))
    bench.broadcast_tensor(t, world)
    bench.barrier(world)
    out[rank] = (m, t.tolist())
    dist.destroy_process_group()


def test_two_rank_reduction_and_broadcast():
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.5          # max over ranks
    assert res[0][1] == res[1][1] == [0.0, 0.0, 0.0]  # rank 0's tensor on every rank


@pytest.mark.parametrize("argv", [["--qat", "--workload", "causal_gqa_det"],     # deterministic
                                  ["--qat", "--workload", "mla_br_causal"],      # D 192
                                  ["--qat", "--bias", "B"],
                                  ["--io", "f16", "--qat"]])
def test_bench_rejects_unsupported_combinations(argv):
    """The option checks run before any GPU work (argparse exits with status 2)."""
    with pytest.raises(SystemExit) as e:
        bench.main(argv + ["--steps", "1", "--warmup", "3"])
    assert e.value.code == 2


def test_bias_bytes_and_traffic_keys():
    w = workloads.WORKLOADS["causal_mha"]
    pairs = bench.visible_pairs(w, None)
    b = torch.zeros((2, 16, 2048, 2048), dtype=torch.bfloat16)
    nbytes = bench.main_kernel_bytes_bias(w, pairs, b)  # fp32 dBias
    # bias at the visible pairs + every fp32 dBias element + Q, dO, K, V, dK, dV, dQ accumulator
    expect = pairs * 2 + b.numel() * 4 + 2 * 2 * 16 * 2048 * 128 * 2 + 2 * (2 * 16 * 2048 * 256 * 2) \
        + 2 * 2 * 16 * 2048 * 128 * 4
    assert nbytes == expect
    t = {"q": torch.zeros(2, 1, 1, 1, dtype=torch.bfloat16), "bias": b}
    assert bench.bias_tag(t) == "bias-B-bf16"
    t["bias"] = torch.zeros((1, 16, 2048, 2048), dtype=torch.float32)
    assert bench.bias_tag(t) == "bias-shared-f32"
    assert bench.bias_tag({"q": t["q"], "qat": True}) == "qat"
    assert bench.bias_tag({"q": t["q"].half()}) == "f16"
    assert bench.bias_tag({"q": t["q"]}) is None


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _json_lines(out: str):
    import json
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _run(cmd):
    import subprocess
    import sys
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable] + cmd, cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return _json_lines(r.stdout)


def _check_reference_line(line, n_gpus):
    assert line["impl"] == "reference" and line["n_gpus"] == n_gpus
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 3 and line["dtype"] == "f64"
    assert line["config"]["workload"] == "tiny_dense"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_prints_one_line():
    """`--impl reference` times the oracle on the host cores and needs no GPU."""
    lines = _run(["bench.py", "--impl", "reference", "--workload", "tiny_dense",
                  "--steps", "1", "--warmup", "3"])
    assert len(lines) == 1
    _check_reference_line(lines[0], 1)


def test_reference_arm_two_ranks_rank0_only():
    """Under the two-process launcher rank 0 alone prints; the other rank exits 0."""
    lines = _run(["-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                  "--master-addr", "127.0.0.1", "--master-port", "29541", "bench.py",
                  "--impl", "reference", "--workload", "tiny_dense", "--gpus", "2",
                  "--steps", "1", "--warmup", "3"])
    assert len(lines) == 1
    _check_reference_line(lines[0], 2)
