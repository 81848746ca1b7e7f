"""CPU checks of bench.py's harness: the replica aggregation over ranks (two
gloo ranks on 127.0.0.1, as torchrun would start them) and the reference
arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_PROGRAM = r"""
import json, os, sys
sys.path.insert(0, os.environ["BENCH_ROOT"])
import torch.distributed as dist
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
import bench
got = bench.max_over_ranks(10.0 + 5.0 * rank, world)
bench.barrier(world)
class Args:
    steps, warmup = 1, 3
ref = bench.run_reference(Args, rank, world) if rank == 1 else "skipped"
dist.destroy_process_group()
print(json.dumps({"rank": rank, "max": got, "ref_is_none": ref is None}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_with_two_gloo_ranks():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), BENCH_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_PROGRAM], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=300)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    by_rank = {d["rank"]: d for d in outs}
    assert by_rank[0]["max"] == by_rank[1]["max"] == 15.0
    assert by_rank[1]["ref_is_none"]  # only rank 0 runs and prints the reference arm


def test_max_over_ranks_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_prints_one_json_line():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "cpu_baseline", "e2e", "config", "dtype"):
        assert key in d
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["value"] > 0


def test_source_hash_ignores_comments_and_layout():
    sys.path.insert(0, ROOT)
    import bench
    code = 'int a = 1; // note\n/* block\n comment */\tconst char *s = "x // y /* z */";\nchar q = \'"\';\n'
    assert bench.code_tokens(code) == 'int a = 1; const char *s = "x // y /* z */"; char q = \'"\';'
    assert bench.code_tokens("a  =\n\n b; // x") == bench.code_tokens("a = b;")
    assert bench.code_tokens("a = b;") != bench.code_tokens("a = c;")
    assert len(bench.source_hash()) == 16
