"""zero_step_amp_noalloc: the mixed-precision step for callers that cannot
allocate device memory (their memory comes from a fixed budget or pool they
do not control, or they run where cudaMalloc/cudaFree are not allowed).  Its
scratch is the library's fixed device array instead of a workspace.

The results must match zero_step_amp with a caller-allocated workspace on
consecutive calls (the fixed array keeps the previous call's contents), both
when this file runs alone in a fresh process (the first call sets the array
up) and after every other test.  This file is named to be collected last.
"""
import gc

import pytest
import torch

from tests._harness import Case
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


def _setup(w, cfg):
    c = Case(w, with_oracle=False)
    c.gsh = [torch.empty(c.plan.shard_len(r), dtype=torch.float32, device="cuda")
             for r in range(w.n_ranks)]
    c.state = Z.amp_state_tensor()
    Z.zero_amp_init(c.state, cfg)
    return c


@pytest.mark.parametrize("numel,N,mode,dtype,op,cfg", [
    ((20000, 37, 4096, 3, 129), 4, "flat", "fp16", "avg",
     Z.AmpConfig(init_scale=1024.0, window=2, hysteresis=2, max_norm=0.05)),
    ((1000, 37, 4096, 3, 129), 3, "round_robin", "bf16", "sum",
     Z.AmpConfig(init_scale=1.0, window=0, hysteresis=1, max_norm=0.0)),
])
def test_noalloc_matches_workspace_entry_point(numel, N, mode, dtype, op, cfg):
    w = W.small(numel, N, mode=mode, align=16, dtype=dtype, op=op, outlier_frac=0.01)
    ref = _setup(w, cfg)
    got = _setup(w, cfg)
    ws = torch.empty(Z.zero_amp_workspace_bytes(ref.plan), dtype=torch.uint8, device="cuda")
    for t in (1, 2):   # two calls in a row on the same fixed scratch
        scale = Z.read_amp_state(ref.state).scale
        g = [W.grads16(w, t, q, "cuda", 0, ref.L, scale=scale) for q in range(N)]
        Z.zero_step_amp(ref.plan, g, op, ref.gsh, ref.master, ref.m, ref.v, ref.full16, None, HP,
                        cfg, ref.state, ws)
        Z.zero_step_amp_noalloc(got.plan, g, op, got.gsh, got.master, got.m, got.v, got.full16,
                                None, HP, cfg, got.state)
        torch.cuda.synchronize()
        sr, sg = Z.read_amp_state(ref.state), Z.read_amp_state(got.state)
        assert (sg.step, sg.skipped, sg.overflow, sg.scale) == (sr.step, sr.skipped, sr.overflow,
                                                                sr.scale)
        assert abs(sg.norm - sr.norm) <= 1e-6 * abs(sr.norm)
        for r in range(N):
            torch.testing.assert_close(got.master[r], ref.master[r], rtol=1e-6, atol=0)
            torch.testing.assert_close(got.m[r], ref.m[r], rtol=1e-6, atol=0)
            torch.testing.assert_close(got.v[r], ref.v[r], rtol=1e-6, atol=0)
        # 16-bit parameters: within one ulp
        a = got.full16.view(torch.int16).long()
        b = ref.full16.view(torch.int16).long()
        key = lambda x: torch.where(x < 0, -(x & 0x7FFF), x)  # noqa: E731
        assert int((key(a) - key(b)).abs().max()) <= 1


def test_noalloc_rejects_steps_beyond_the_fixed_scratch():
    """A group of 300M elements needs more than 2 MiB of scratch: the call
    fails with a clear message and launches nothing."""
    plan = Z.zero_plan_partitions([300_000_000], 1, "flat", 16)
    assert Z.zero_amp_workspace_bytes(plan) > (2 << 20)
    state = Z.amp_state_tensor()
    Z.zero_amp_init(state, Z.AmpConfig())
    before = Z.zero_launch_count()
    big = 1 << 30   # aligned stand-in addresses; nothing is launched
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_step_amp_noalloc(plan, [big], "sum", [big], [big], [big], [big], None, None, HP,
                                Z.AmpConfig(), state, dtype=Z.ZERO_FP16)
    assert e.value.status == Z.ZERO_ERR_INVALID
    assert "fixed scratch" in str(e.value) and "zero_step_amp" in str(e.value)
    assert Z.zero_launch_count() == before


def test_noalloc_call_allocates_no_device_memory():
    """After a first call (which may load the library's device code on this
    device and commit the fixed scratch), further calls leave the device's
    free memory and torch's allocation counters unchanged."""
    w = W.small((20000, 37, 4096, 3, 129), 4, mode="flat", align=16, dtype="bf16", op="avg")
    cfg = Z.AmpConfig(init_scale=1.0, window=0, hysteresis=1, max_norm=1.0)
    c = _setup(w, cfg)
    g = [W.grads16(w, 1, q, "cuda", 0, c.L) for q in range(4)]

    def call():
        Z.zero_step_amp_noalloc(c.plan, g, "avg", c.gsh, c.master, c.m, c.v, c.full16, None, HP,
                                cfg, c.state)
    call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0
    for k in ("allocation.all.allocated", "segment.all.allocated", "num_alloc_retries"):
        assert stats1.get(k, 0) == stats0.get(k, 0), k
    assert Z.read_amp_state(c.state).step == 4
