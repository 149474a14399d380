"""The N > 1 path on the CPU with two gloo ranks.

bench.py runs one independent replica per GPU (requests and kv heads are independent, so the path
needs no collective) and reports the slowest rank's step time.  These tests cover that host logic
and the one exchange step a split of a long context across GPUs would need: an all-gather of the
ranks' partial (out, lse) followed by the split-result merge (ZipFusion §IV.B), here with the oracle.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from oracle import zf_oracle as O


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, fn, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, fn(rank, world)))
    finally:
        dist.destroy_process_group()


def run_ranks(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, fn, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return [out[r] for r in range(world)]


def _rand_bits(rng, shape, std=1.0):
    x = (rng.standard_normal(shape) * std).astype(np.float32)
    return ((x.view(np.uint32) + 0x8000) >> 16).astype(np.uint16)


def _slowest(rank, world):
    return bench.max_over_ranks(10.0 + rank, torch.device("cpu"))


def test_step_time_is_the_slowest_rank():
    assert run_ranks(_slowest) == [11.0, 11.0]


def test_replica_request_sharding_covers_the_batch():
    for B in (1, 2, 5, 64, 127):
        for world in (1, 2, 3, 8):
            got = [bench.replica_requests(B, r, world) for r in range(world)]
            assert sorted(sum(got, [])) == list(range(B))
            assert max(map(len, got)) - min(map(len, got)) <= 1


def _token_split(rank, world):
    rng = np.random.default_rng(0)                  # same data on every rank
    q = O.bf16_to_f64(_rand_bits(rng, (128,)))
    K = O.bf16_to_f64(_rand_bits(rng, (901, 128), 2.0))
    V = O.bf16_to_f64(_rand_bits(rng, (901, 128)))
    cuts = np.linspace(0, 901, world + 1).astype(int)
    o, l, _ = O.attention_one(q, K[cuts[rank]:cuts[rank + 1]], V[cuts[rank]:cuts[rank + 1]], 0.09)
    mine = torch.tensor(np.concatenate([o, [l]]), dtype=torch.float64)
    parts = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(parts, mine)
    mo, ml = O.merge_partials([p[:128].numpy() for p in parts], [float(p[128]) for p in parts])
    ref, ref_l, _ = O.attention_one(q, K, V, 0.09)
    return float(np.abs(mo - ref).max()), abs(ml - ref_l)


def test_token_split_exchange_then_merge_equals_unsplit():
    for err, lerr in run_ranks(_token_split):
        assert err < 1e-12 and lerr < 1e-12


def _batch_shard(rank, world):
    rng = np.random.default_rng(1)
    B = 5
    q = _rand_bits(rng, (B, 4, 128))
    ks = [_rand_bits(rng, (17 + 9 * b, 2, 128), 2.0) for b in range(B)]
    vs = [_rand_bits(rng, (17 + 9 * b, 2, 128)) for b in range(B)]
    mine = bench.replica_requests(B, rank, world)
    out, lse = O.attention_dense(q[mine], [ks[b] for b in mine], [vs[b] for b in mine], 0.1)
    full, full_lse = O.attention_dense(q, ks, vs, 0.1)
    return bool((out == full[mine]).all() and (lse == full_lse[mine]).all())


def test_replicas_on_disjoint_requests_reproduce_the_full_batch():
    assert run_ranks(_batch_shard) == [True, True]


STUB = """
import json, sys
import torch
import torch.distributed as dist
dist.init_process_group("gloo")
r, w = dist.get_rank(), dist.get_world_size()
t = torch.tensor([10.0 + r])
dist.all_reduce(t, op=dist.ReduceOp.MAX)
if r == 0:
    print(json.dumps({"world": w, "max": float(t.item()), "args": sys.argv[1:]}), flush=True)
dist.destroy_process_group()
"""


def test_launcher_starts_one_rank_per_gpu(tmp_path):
    """bench.py --gpus N run without torchrun starts N ranks itself (torch.distributed.run on
    127.0.0.1); here the ranks are gloo processes running a stand-in script."""
    import json
    stub = tmp_path / "stub.py"
    stub.write_text(STUB)
    res = bench.launch_ranks(2, ["--steps", "3"], script=str(stub), capture_output=True)
    assert res.returncode == 0, res.stderr[-2000:]
    line = [x for x in res.stdout.splitlines() if x.startswith("{")][-1]
    got = json.loads(line)
    assert got == {"world": 2, "max": 11.0, "args": ["--steps", "3"]}


def test_main_hands_gpus_above_one_to_the_launcher(monkeypatch):
    seen = {}

    class Done:
        returncode = 0

    def fake(n, argv, script=None, capture_output=False):
        seen["n"], seen["argv"] = n, list(argv)
        return Done()
    monkeypatch.setattr(bench, "launch_ranks", fake)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr("sys.argv", ["bench.py", "--gpus", "4", "--steps", "5"])
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert e.value.code == 0 and seen == {"n": 4, "argv": ["--gpus", "4", "--steps", "5"]}
