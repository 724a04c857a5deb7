"""Host logic of bench.py without a GPU: max-over-ranks timing and barriers
on a 2-rank gloo group, and the reference arm's JSON line."""
import json
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    got = bench.max_over_ranks(dist, 1.5 + r)  # rank 1 is the slow one
    bench.barrier(dist)
    dist.destroy_process_group()
    q.put((r, got))


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, 2.5), (1, 2.5)]


def test_reference_arm_line(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3",
                       "--ref-budget", "1"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in line
    assert line["impl"] == "reference" and line["unit"] == "params/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_other_ranks_do_nothing(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3",
                       "--ref-budget", "1"]) == 0
    assert capsys.readouterr().out.strip() == ""


def test_warmup_floor():
    sys.path.insert(0, ROOT)
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_step_bytes():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.step_bytes(109482240, 8) == 4598254080
    assert bench.step_bytes(1053760, 4) == 35827840
    assert bench.step_bytes(212336640, 8, n16_out=2) == 44 * 212336640


def test_headline_and_per_config_groups():
    """The default line times the LLaMA-7B rank-0 shard (42 B per element over
    842,301,952 elements, 50M-element buckets: 17 launches); per_config names
    every other group once, the tiny group in both regimes."""
    sys.path.insert(0, ROOT)
    import bench
    from zero_sharded_optimizer_flatten_gb300 import workloads as W
    w = W.WORKLOADS[bench.WORKLOAD]
    assert bench.WORKLOAD == "llama7b_rank0" and w.mask == 1 and w.bucket_elems == 50_000_000
    S = 842_301_952
    assert bench.step_bytes(S, w.n_ranks) == 35_376_681_984
    assert -(-S // w.bucket_elems) == 17
    keys = [k for k, *_ in bench.PER_CONFIG]
    assert len(set(keys)) == len(keys)
    groups = {wk for _, wk, _, _ in bench.PER_CONFIG}
    assert groups == {"tiny_mlp", "bert_base", "toy_rr", "llama13b_layer"}
    assert all(wk in W.WORKLOADS for wk in groups)
    assert {k for k in keys if k.startswith("tiny_mlp/")} == {"tiny_mlp/back_to_back",
                                                              "tiny_mlp/l2_flushed"}
    flushed = [opt for k, _, _, opt in bench.PER_CONFIG if k == "tiny_mlp/l2_flushed"][0]
    assert flushed.get("flush_l2") and flushed["warmup"] >= 3


def test_host_available_bytes():
    sys.path.insert(0, ROOT)
    import bench
    free = bench.host_available_bytes()
    assert free is None or free > 0


def test_zero3_layer_states_fit_free_memory(monkeypatch):
    """The 40-layer ZeRO-3 record keeps 40 distinct layer states when the
    device has room (about 3 GB each for the 212M-element layer) and cycles
    fewer, a divisor of 40, when it does not."""
    sys.path.insert(0, ROOT)
    import torch

    import bench
    from zero_sharded_optimizer_flatten_gb300 import workloads as W
    w = W.WORKLOADS["llama13b_layer"]
    for free_gb, want in ((275, 40), (100, 20), (40, 8), (5, 1)):
        monkeypatch.setattr(torch.cuda, "mem_get_info",
                            lambda dev=None, f=free_gb: (f * 10 ** 9, 280 * 10 ** 9))
        assert bench.zero3_layer_states(w, None, 40) == want, free_gb
