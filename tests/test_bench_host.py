"""Host-side logic of bench.py that needs no GPU: the multi-rank timing
reduction (world size 2 over gloo on CPU) and the reference arm's behaviour
on non-zero ranks."""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, values, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank])
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        values = [3.5, 7.25]
        procs = [ctx.Process(target=_worker, args=(r, 2, port, values, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == out[1] == 7.25


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5) == 1.5


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_summary_puts_the_five_configurations_last():
    """The JSON line ends with a short per-workload summary whose last five
    entries are the problem's five configurations (the part of a long line a
    tail shows)."""
    import bench
    per = {n: {"ms": 1.0, "roofline_frac": 0.5, "elements_per_s": 2.0}
           for n in ("s6_bidir", "affine_small", "s6_fp32_bwd", "affine_large", "s6_fp32",
                     "s6_bf16", "s6_bf16_layer")}
    per["s6_fp32"]["cpu_baseline"] = {"value": 8.0, "value_1_thread": 1.0, "cores": 16,
                                      "host_cores": 16}
    out = bench.config_summary(per, {"cpu_baseline": {"value": 3.0, "cores": 1, "host_cores": 16}})
    assert list(out)[-5:] == ["affine_small", "affine_large", "s6_fp32", "s6_bf16", "s6_bidir"]
    assert out["s6_fp32"]["oracle_elem_per_s"] == {"1_thread": 1.0, "all_cores": 8.0, "cores": 16}
    assert out["affine_large"]["oracle_elem_per_s"]["1_thread"] == 3.0
    r = bench.round_floats({"a": 1.23456789, "b": [7, 2.0000001], "c": "x"})
    assert r == {"a": 1.2346, "b": [7, 2.0], "c": "x"}
