"""The multi-rank path of bench.py on CPU (gloo, world_size 2).

With N > 1 every rank runs an independent replica of the workload (the work
items are independent; there is no data-path collective): the step time is the
max over ranks, the bytes are summed, and only rank 0 prints.  These tests run
the rank helpers and the reference arm under two gloo processes on 127.0.0.1.
"""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    times = [0.25, 0.75]
    mx = bench.max_over_ranks(times[rank], w, "cpu")
    sm = bench.sum_over_ranks(1000.0 * (rank + 1), w, "cpu")
    bench.barrier(w)
    q.put((rank, r, w, lr, mx, sm))
    dist.destroy_process_group()


def test_rank_helpers_take_max_time_and_sum_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, w, lr, mx, sm in got:
        assert (r, w, lr) == (rank, 2, rank)
        assert mx == 0.75 and sm == 3000.0


def test_reference_arm_prints_once_under_two_ranks(tmp_path):
    # launch bench.py --impl reference as two ranks (env as torchrun sets it);
    # rank 0 prints exactly one JSON line, rank 1 exits 0 without output
    outs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT="1")
        outs.append(subprocess.run(
            [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
             "--steps", "1", "--warmup", "0", "--workload", "1"],
            cwd=ROOT, env=env, capture_output=True, text=True, timeout=600))
    assert all(o.returncode == 0 for o in outs), [o.stderr[-2000:] for o in outs]
    lines0 = [l for l in outs[0].stdout.splitlines() if l.startswith("{")]
    assert len(lines0) == 1 and outs[1].stdout.strip() == ""
    d = json.loads(lines0[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_kernel_hash_ignores_comments_but_not_code():
    # the committed traffic capture is keyed to the split kernel's code:
    # comment and layout edits keep the key, any code edit changes it
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    src = 'int a = 1;  // note\n/* block\n comment */ const char* s = "// kept";\nchar q = \'"\';\n'
    assert bench.code_tokens(src) == 'int a = 1; const char* s = "// kept"; char q = \'"\';'
    assert bench.code_tokens(src.replace("// note", "// other note")) == bench.code_tokens(src)
    assert bench.code_tokens(src.replace("a = 1", "a = 2")) != bench.code_tokens(src)
    with open(os.path.join(ROOT, "profiles", "split_kv_traffic.json")) as f:
        assert len(json.load(f)["source_hash"]) == len(bench.kernel_source_hash()) == 16
