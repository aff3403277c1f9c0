"""The data-parallel harness of bench.py on CPU: two gloo ranks.

Checks the pieces a multi-GPU run relies on without touching a GPU: the
environment parsing, the max-over-ranks reduction of the timed region, the
whole-job aggregate (all ranks' tokens over the slowest rank's time), that
each rank draws its own token batch while the weights stay shared, and that
the reference arm does its work on rank 0 only."""
import argparse
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, loc = bench.dist_env()
        # rank r timed 1 + r seconds: every rank must see the slowest
        sec_max = bench.max_over_ranks(1.0 + r, w)
        lay = synth.layer("tiny")
        x, lg = bench.make_inputs(lay, bench.shard_seed(0, r))
        w1 = lay.w1_expert(0)
        # the reference arm returns at once on ranks other than 0
        args = argparse.Namespace(workload="tiny", seed=0, ref_tokens=2, warmup=3, steps=1)
        ref_ret = bench.reference(args) if r != 0 else None
        dist.barrier()
        q.put(dict(rank=r, world=w, local=loc, sec_max=sec_max,
                   x_sum=float(np.asarray(x, dtype=np.float64).sum()),
                   lg_sum=float(np.asarray(lg, dtype=np.float64).sum()),
                   w1_sum=float(np.asarray(w1, dtype=np.float64).sum()), ref_ret=ref_ret))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res = sorted(res, key=lambda d: d["rank"])
    assert [d["rank"] for d in res] == [0, 1] and all(d["world"] == 2 for d in res)
    assert [d["local"] for d in res] == [0, 1]
    assert all(d["sec_max"] == 2.0 for d in res)
    # data parallel: different token batches, the same weights
    assert res[0]["x_sum"] != res[1]["x_sum"] and res[0]["lg_sum"] != res[1]["lg_sum"]
    assert res[0]["w1_sum"] == res[1]["w1_sum"]
    assert res[1]["ref_ret"] is None


def test_aggregate_and_seeds():
    sys.path.insert(0, ROOT)
    import bench
    # 4 ranks x 65536 tokens x 10 steps over the slowest rank's 2 s
    assert bench.aggregate(65536, 10, 4, 2.0) == 65536 * 10 * 4 / 2.0
    seeds = {bench.shard_seed(7, r) for r in range(8)}
    assert len(seeds) == 8 and bench.shard_seed(7, 0) == 7
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_source_hash_ignores_comments(tmp_path, monkeypatch):
    """The kernel-source hash that keys bench.py's recorded ncu traffic: the
    same for code that differs only in // comments and blank lines, different
    for a changed statement."""
    sys.path.insert(0, ROOT)
    import bench
    csrc = tmp_path / "nvfp4_w4a4_moe_top_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))

    def sha_of(text):
        (csrc / "k.cu").write_text(text)
        return bench.src_sha("k.cu")

    base = sha_of("int f(int x) {\n  return x + 1;\n}\n")
    assert sha_of("// a comment\nint f(int x) {  // trailing\n\n  return x + 1;   \n}\n") == base
    assert sha_of("int f(int x) {\n  return x + 2;\n}\n") != base


def test_reference_arm_line(capsys, monkeypatch):
    """The reference arm (the oracle on the host cores) on one process: one
    JSON line with the native arm's metric, unit and config, its own
    cpu_baseline and an e2e entry without copies; with no explicit sample
    size it takes whole 256-token samples of the tiny layer."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    import synth
    for v in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(v, raising=False)
    args = argparse.Namespace(workload="tiny", seed=0, ref_tokens=None, warmup=3, steps=1)
    bench.reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    lay = synth.layer("tiny")
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["config"] == bench.config_of("tiny", lay, 1)
    assert line["steps"] == 1 and line["warmup"] == 3 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["sample"].startswith("256 consecutive tokens")
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0

