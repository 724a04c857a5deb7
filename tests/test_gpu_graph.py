"""Steps captured in a CUDA graph and replayed: the bucketed fused step (a
chain of launches where every launch after a run's first starts early) and
the mixed-precision step must give the oracle's results when replayed from
a graph, as they do when launched from the host (the bench times graph
replays)."""
import gc

import pytest
import torch

from tests._harness import Case, hp_oracle
from tests.test_gpu_amp import AmpCase
from zero_sharded_optimizer_flatten_gb300 import workloads as W
from zero_sharded_optimizer_flatten_gb300 import zero as Z

pytestmark = pytest.mark.gpu

HP = Z.AdamW()


@pytest.fixture(autouse=True)
def _cuda_cleanup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _capture(fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("numel,N,mode,A,dtype,bucket", [
    ((200000, 37, 90001, 3, 129), 4, "flat", 16, "bf16", 20000),
    ((200000, 37, 90001, 3, 129), 8, "flat", 2, "fp16", 7000),
    (tuple(5 + (k * 7919) % 3001 for k in range(700)), 3, "round_robin", 1, "fp16", 400000),
])
def test_bucketed_step_replayed_from_a_graph(numel, N, mode, A, dtype, bucket):
    w = W.small(numel, N, mode=mode, align=A, dtype=dtype, op="avg")
    c = Case(w)
    grads = [c.grads(t) for t in (1, 2, 3)]
    n0 = Z.zero_launch_count()

    def three_steps():
        for t in (1, 2, 3):
            Z.zero_step(c.plan, grads[t - 1], "avg", c.master, c.m, c.v, c.full16, None, HP, t,
                        bucket_elems=bucket)
    graph = _capture(three_steps)
    assert Z.zero_launch_count() - n0 >= 6          # several launches per step
    for rep in range(2):                            # replaying applies steps 1..3 again
        graph.replay()
        for t in (1, 2, 3):
            c.oracle_step(grads[t - 1], t, hp_oracle(HP))
        torch.cuda.synchronize()
        c.compare(f"replay {rep}")


def test_mixed_precision_step_replayed_from_a_graph():
    w = W.small((200000, 37, 90001, 3, 129), 4, mode="flat", align=16, dtype="fp16", op="avg",
                outlier_frac=0.01)
    cfg = Z.AmpConfig(init_scale=1.0, window=0, hysteresis=1, max_norm=0.05)
    c = AmpCase(w, cfg, bucket=30000)
    grads = [c.grads_scaled(t, 1.0) for t in (1, 2, 3)]

    def three_steps():
        for g in grads:
            c.gpu_step(g)
    graph = _capture(three_steps)
    graph.replay()
    for g in grads:
        c.oracle_step_amp(g)
    torch.cuda.synchronize()
    c.compare_state("after the replay")
    c.compare("mixed precision from a graph")
    assert c.ost.step == 3
