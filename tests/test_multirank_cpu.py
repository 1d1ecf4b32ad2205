"""The multi-rank path of bench.py on the CPU: two gloo ranks on 127.0.0.1.

Each rank runs one full replica (weak scaling); the only collectives are the
timing barrier and the max over ranks of the elapsed time.  The reference arm
runs and prints on rank 0 only; the other ranks return without work.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout
from types import SimpleNamespace

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    got = bench.max_over_ranks(10.0 + 3.0 * rank, world)
    args = SimpleNamespace(workload="prefill_s4k_gqa_bf16", warmup=1, steps=1, ref_rows=2)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, world, rank)
    bench.barrier(world)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"max": got, "stdout": buf.getvalue()}, f)


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    assert r0["max"] == r1["max"] == 13.0
    assert r1["stdout"] == ""
    line = json.loads(r0["stdout"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == world and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
