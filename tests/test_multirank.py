"""The N > 1 path of bench.py on CPU: two gloo ranks run replicas (each its own batch, drawn with a
rank-dependent seed), agree on the slowest rank's step time, and report the whole job's tokens/s;
the reference arm prints from rank 0 only."""
import argparse
import json
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        import bench
        import dsv4_inputs as I
        cfg = bench.rank_config(I.SMALL_CONFIGS["small_c4_bf16"], rank)
        st = I.make_step(cfg)
        ms = 1.0 + 0.5 * rank  # rank 1 is the slower one
        slowest = bench.max_over_ranks(ms, world, "cpu")
        value = bench.job_tokens_per_s(cfg.T, world, slowest)
        np.save(os.path.join(out_dir, f"q{rank}.npy"), np.asarray(st.q))
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "value": value, "T": cfg.T, "seed": cfg.seed}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replica_ranks_on_gloo(tmp_path):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    r = [json.load(open(tmp_path / f"r{k}.json")) for k in range(2)]
    assert r[0]["slowest"] == r[1]["slowest"] == 1.5
    assert r[0]["value"] == r[1]["value"] == pytest.approx(2 * r[0]["T"] / 1.5e-3)
    assert r[0]["seed"] != r[1]["seed"]
    q0, q1 = (np.load(tmp_path / f"q{k}.npy") for k in range(2))
    assert q0.shape == q1.shape and not np.array_equal(q0, q1)  # each rank decodes its own batch


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5
    assert bench.job_tokens_per_s(32, 1, 2.0) == pytest.approx(16000.0)


def test_reference_arm_prints_from_rank_0_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(argparse.Namespace(config="small_c4_bf16", steps=1, warmup=0))
    assert capsys.readouterr().out == ""
