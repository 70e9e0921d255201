"""Host logic of bench.py that needs no GPU: the reference arm's JSON line
(the CPU oracle on a bounded sample) and the multi-rank reduction (max over
ranks) under torch.distributed with the gloo backend, world size 2."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_bf16", "--steps", "1", "--ref-tokens", "2"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny_bf16"
    assert 1 <= d["cpu_baseline"]["cores"] <= os.cpu_count()
    # a step of this arm is the sampled step that was timed, not the full batch
    assert d["tokens_per_step"] == 2 and d["steps"] == 1
    assert abs(d["ms_per_step"] - 2 / d["value"] * 1e3) <= 1e-6 * d["ms_per_step"]
    assert d["extrapolated_ms_per_full_batch"] > d["ms_per_step"]


def test_reference_arm_under_torchrun_prints_once():
    # two ranks: rank 0 alone times the oracle and prints; rank 1 exits 0
    port = 29000 + os.getpid() % 1000
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                          "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                          "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                          "--impl", "reference", "--gpus", "2", "--workload", "tiny_bf16",
                          "--steps", "1", "--ref-tokens", "2"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method="env://")
    bench._barrier(world)
    v = bench._max_over_ranks(1.5 + rank, world, "cpu")
    q.put((rank, bench._dist(), v))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    assert all(v == 2.5 for _, _, v in res)          # both ranks see the slowest time
    assert res[1][1] == (2, 1, 1)                      # (world size, rank, local rank)


def test_profile_commands_run_committed_files_with_valid_options():
    # every bench command a profile summary names parses with bench.py's own
    # options and names a workload the generators define
    import glob
    import re
    import shlex
    sys.path.insert(0, ROOT)
    import bench
    ap = bench.build_parser()
    seen = 0
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(path).read().replace("\\\n", " ")
        for cmd in re.findall(r"python bench\.py[^\n`]*", text):
            argv = shlex.split(cmd)[2:]
            ap.parse_args(argv)                      # exits on an unknown option
            seen += 1
    assert seen >= 5
