"""The autograd-driven engine: gradient hooks fill each virtual rank's flat
replica, full buckets are reduce-scattered during the backward pass (on a
side stream with overlap_comm), step() updates and gathers.  The engine's
replicas must be the gradients torch computes, and its update must be the
oracle's step on those replicas."""
import gc

import numpy as np
import pytest
import torch

import oracle
from tests._harness import assert_16_close, assert_fp32_close, f32, hp_oracle, u16
from zero_sharded_optimizer_flatten_gb300 import zero as Z
from zero_sharded_optimizer_flatten_gb300.engine import ZeroEngine

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda_cleanup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _mlp(dtype, seed=0):
    torch.manual_seed(seed)
    layers = []
    for _ in range(2):
        layers += [torch.nn.Linear(256, 1024), torch.nn.GELU(), torch.nn.Linear(1024, 256)]
    layers += [torch.nn.Linear(256, 10)]
    return torch.nn.Sequential(*layers).to("cuda", dtype)


def _batch(q, t, dtype):
    g = torch.Generator(device="cuda")
    g.manual_seed(1000 * t + q)
    return torch.randn(32, 256, generator=g, device="cuda", dtype=torch.float32).to(dtype)


def _loss(model, x):
    return model(x).float().pow(2).mean()


@pytest.mark.parametrize("bucket,overlap,mode", [(100_000, True, "flat"), (100_000, False, "flat"),
                                                 (0, True, "flat"), (50_000, True, "round_robin")])
def test_engine_matches_torch_grads_and_oracle_step(bucket, overlap, mode):
    dtype = torch.bfloat16
    N = 4
    model = _mlp(dtype)
    names = [n for n, _ in model.named_parameters()]
    hp = Z.AdamW()
    eng = ZeroEngine(model.parameters(), N, mode=mode, align=16, op="avg", hparams=hp,
                     bucket_elems=bucket, overlap_comm=overlap)
    plan = eng.plan
    mode_c = oracle.FLAT if mode == "flat" else oracle.ROUND_ROBIN
    # oracle state from the engine's initial parameters
    p16 = u16(eng.flat16)
    om, omm, ov = [], [], []
    for r in range(N):
        seg = oracle.segments(eng.numel, N, mode_c, 16, r)
        S = int(seg[:, 4].sum()) if len(seg) else 0
        x = np.zeros(S, np.float32)
        for k, toff, foff, soff, ln in seg:
            x[soff:soff + ln] = oracle.to_f32(p16[foff:foff + ln], oracle.BF16)
        om.append(x)
        omm.append(np.zeros(S, np.float32))
        ov.append(np.zeros(S, np.float32))
    ofull = np.zeros(plan.padded, np.uint16)
    for t in (1, 2, 3):
        for q in range(N):
            x = _batch(q, t, dtype)
            # the expected gradients: a plain backward of the same model (the
            # engine's hooks ignore backward passes outside eng.backward)
            _loss(model, x).backward()
            expect = torch.cat([p.grad.reshape(-1) for p in model.parameters()])
            model.zero_grad(set_to_none=True)
            eng.backward(_loss(model, x), q)
            torch.cuda.synchronize()
            assert torch.equal(eng.grads[q][:plan.phi], expect), (t, q)
            assert all(p.grad is None for p in model.parameters())   # released
        replicas = [u16(g) for g in eng.grads]
        eng.step()
        oracle.step(eng.numel, N, mode_c, 16, oracle.BF16, oracle.AVG, replicas, om, omm, ov, ofull,
                    None, hp_oracle(hp), t)
        torch.cuda.synchronize()
        for r in range(N):
            assert_fp32_close(f32(eng.master[r]), om[r], f"t={t} master[{r}]")
            assert_fp32_close(f32(eng.v[r]), ov[r], f"t={t} v[{r}]")
        assert_16_close(u16(eng.flat16), ofull, f"t={t} flat16")
        # the model's parameters are views of the gathered buffer
        flat_again = torch.cat([p.detach().reshape(-1) for p in model.parameters()])
        assert torch.equal(flat_again, eng.flat16[:plan.phi])
    if bucket and overlap:
        assert eng.launched_during_backward > 0
    assert names


def test_engine_overlap_does_not_change_results():
    dtype = torch.bfloat16
    a, b = _mlp(dtype), _mlp(dtype)
    ea = ZeroEngine(a.parameters(), 4, bucket_elems=0, overlap_comm=False)
    eb = ZeroEngine(b.parameters(), 4, bucket_elems=60_000, overlap_comm=True)
    for t in (1, 2):
        for q in range(4):
            x = _batch(q, t, dtype)
            ea.backward(_loss(a, x), q)
            eb.backward(_loss(b, x), q)
        ea.step()
        eb.step()
    torch.cuda.synchronize()
    assert torch.equal(ea.flat16, eb.flat16)
    for r in range(4):
        assert torch.equal(ea.master[r], eb.master[r])


def test_engine_requires_every_rank():
    model = _mlp(torch.bfloat16)
    eng = ZeroEngine(model.parameters(), 2)
    eng.backward(_loss(model, _batch(0, 1, torch.bfloat16)), 0)
    with pytest.raises(RuntimeError):
        eng.step()
    with pytest.raises(RuntimeError):
        eng.backward(_loss(model, _batch(0, 1, torch.bfloat16)), 0)


@pytest.mark.parametrize("offload,overlap,dtype", [("cpu", True, torch.bfloat16),
                                                   ("cpu", False, torch.float16),
                                                   ("host_state", True, torch.bfloat16)])
def test_engine_offload_modes_equal_the_device_engine(offload, overlap, dtype):
    """offload_optimizer to the host: the CPU optimizer (reductions into pinned
    host shards, host AdamW + cast, gather) and the host-resident state that
    the GPU kernels update across the link both give the device engine's
    parameters and state bit for bit."""
    a, b = _mlp(dtype), _mlp(dtype)
    ea = ZeroEngine(a.parameters(), 4, bucket_elems=60_000, overlap_comm=overlap)
    eb = ZeroEngine(b.parameters(), 4, bucket_elems=60_000, overlap_comm=overlap,
                    offload=offload, host_threads=3)
    assert all(not x.is_cuda and x.is_pinned() for x in eb.master + eb.m + eb.v)
    if offload == "cpu":
        assert all(x.is_pinned() for x in eb.grad_shards + eb.shard16)
    for t in (1, 2, 3):
        for q in range(4):
            x = _batch(q, t, dtype)
            ea.backward(_loss(a, x), q)
            eb.backward(_loss(b, x), q)
        ea.step()
        eb.step()
    torch.cuda.synchronize()
    assert torch.equal(ea.flat16, eb.flat16)
    for r in range(4):
        for xa, xb in ((ea.master[r], eb.master[r]), (ea.m[r], eb.m[r]), (ea.v[r], eb.v[r])):
            assert torch.equal(xa.cpu(), xb.cpu())


@pytest.mark.parametrize("offload", ["host_state", "cpu"])
def test_engine_mixed_precision_with_offload(offload):
    """amp with the state in host memory, updated by the GPU across the link
    or by host threads after the device's decision: the same decisions and
    updates as the device-resident engine, bit for bit (fp16, a loss scale
    that overflows at first, clipping)."""
    cfg = Z.AmpConfig(init_scale=2.0 ** 24, min_scale=1.0, window=20, hysteresis=1,
                      max_norm=1.0)
    a, b = _mlp(torch.float16), _mlp(torch.float16)
    ea = ZeroEngine(a.parameters(), 4, bucket_elems=60_000, amp=cfg)
    eb = ZeroEngine(b.parameters(), 4, bucket_elems=60_000, amp=cfg, offload=offload,
                    host_threads=3)
    for t in range(1, 8):
        for q in range(4):
            x = _batch(q, t, torch.float16)
            ea.backward(_loss(a, x), q)
            eb.backward(_loss(b, x), q)
        ea.step()
        eb.step()
    torch.cuda.synchronize()
    sa, sb = ea.amp_status(), eb.amp_status()
    assert bytes(sa) == bytes(sb) and sa.skipped >= 1
    assert torch.equal(ea.flat16, eb.flat16)
    for r in range(4):
        assert torch.equal(ea.master[r].cpu(), eb.master[r])
        assert torch.equal(ea.v[r].cpu(), eb.v[r])


def test_engine_offload_arguments():
    with pytest.raises(ValueError):
        ZeroEngine(_mlp(torch.bfloat16).parameters(), 2, offload="nvme")


@pytest.mark.parametrize("amp,offload", [(False, None), (True, None), (False, "cpu"),
                                         (False, "host_state"), (True, "host_state")])
def test_engine_checkpoint_resume_is_bit_identical(amp, offload):
    """state_dict() after three iterations, load_state_dict() into a fresh
    engine over a differently initialised model, two more iterations: the
    parameters and the optimizer (and mixed-precision) state equal those of
    five uninterrupted iterations bit for bit."""
    dtype = torch.float16 if amp else torch.bfloat16
    cfg = (Z.AmpConfig(init_scale=2.0 ** 24, min_scale=1.0, window=2, hysteresis=1,
                       max_norm=1.0) if amp else None)

    def engine(model):
        return ZeroEngine(model.parameters(), 4, bucket_elems=60_000, amp=cfg, offload=offload)

    def iterate(eng, model, t):
        for q in range(4):
            eng.backward(_loss(model, _batch(q, t, dtype)), q)
        eng.step()

    a = _mlp(dtype)
    ea = engine(a)
    for t in range(1, 6):
        iterate(ea, a, t)
    b = _mlp(dtype)
    eb = engine(b)
    for t in range(1, 4):
        iterate(eb, b, t)
    sd = eb.state_dict()
    c = _mlp(dtype, seed=5)
    ec = engine(c)
    with pytest.raises(ValueError):
        ZeroEngine(_mlp(dtype).parameters(), 2).load_state_dict(sd)
    ec.load_state_dict(sd)
    for t in range(4, 6):
        iterate(ec, c, t)
    torch.cuda.synchronize()
    assert torch.equal(ea.flat16, ec.flat16)
    for r in range(4):
        for x, y in ((ea.master[r], ec.master[r]), (ea.m[r], ec.m[r]), (ea.v[r], ec.v[r])):
            assert torch.equal(x.cpu(), y.cpu())
    if amp:
        assert torch.equal(ea.amp_state, ec.amp_state)
        assert Z.read_amp_state(ea.amp_state).skipped >= 1
    assert ec.step_count == ea.step_count == 5
