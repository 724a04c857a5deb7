"""End to end: a model trains through the autograd-driven engine.

A bf16 student MLP learns a fixed random teacher (mean squared error) for 60
iterations with 4 virtual ranks, each running forward and backward on its own
micro-batch through ZeroEngine (bucketed reduce-scatter overlapped with the
backward pass, then AdamW + cast + all-gather in the library).  The reference
is the same student trained by torch: per-rank bf16 gradients summed in rank
order in fp32 and divided by 4, `torch.optim.AdamW` on fp32 master copies,
parameters rounded back to bf16 after every step.  torch's AdamW rounds its
moment update differently (a lerp), so the two runs are compared as loss
curves, not bit for bit; the bit-level parity of each piece is covered by the
engine and parity tests.

The second test runs the engine's mixed-precision form: an fp16 model with a
dynamic loss scale, overflow skips and clipping, checked step by step against
zero_step_amp on the engine's own replicas, and for convergence.
"""
import copy
import gc

import pytest
import torch

from zero_sharded_optimizer_flatten_gb300 import zero as Z
from zero_sharded_optimizer_flatten_gb300.engine import ZeroEngine

pytestmark = pytest.mark.gpu

N = 4
STEPS = 60


@pytest.fixture(autouse=True)
def _cuda_cleanup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _mlp(seed, dtype):
    torch.manual_seed(seed)
    return torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.GELU(),
                               torch.nn.Linear(256, 256), torch.nn.GELU(),
                               torch.nn.Linear(256, 8)).to("cuda", dtype)


def _micro_batch(q, t):
    g = torch.Generator(device="cuda")
    g.manual_seed(7919 * t + q)
    return torch.randn(64, 64, generator=g, device="cuda")


def test_engine_trains_like_torch_adamw():
    teacher = _mlp(123, torch.float32)
    student = _mlp(1, torch.bfloat16)
    ref = copy.deepcopy(student)
    masters = [p.detach().float().clone() for p in ref.parameters()]
    opt = torch.optim.AdamW(masters, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01,
                            foreach=False)
    eng = ZeroEngine(student.parameters(), N, mode="flat", align=16, op="avg",
                     hparams=Z.AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01), bucket_elems=20_000,
                     overlap_comm=True)

    def loss_of(model, x):
        with torch.no_grad():
            y = teacher(x)
        return (model(x.to(torch.bfloat16)).float() - y).pow(2).mean()

    curve_eng, curve_ref = [], []
    for t in range(STEPS):
        xs = [_micro_batch(q, t) for q in range(N)]
        # the engine: each virtual rank's backward feeds its gradient replica
        le = 0.0
        for q in range(N):
            loss = loss_of(student, xs[q])
            eng.backward(loss, q)
            le += loss.item() / N
        eng.step()
        curve_eng.append(le)
        # the reference: the same per-rank gradients, averaged in rank order
        lr_ = 0.0
        acc = None
        for q in range(N):
            ref.zero_grad(set_to_none=True)
            loss = loss_of(ref, xs[q])
            loss.backward()
            lr_ += loss.item() / N
            g = [p.grad.float() for p in ref.parameters()]
            acc = g if acc is None else [a + b for a, b in zip(acc, g)]
        for mst, a in zip(masters, acc):
            mst.grad = a / N
        opt.step()
        with torch.no_grad():
            for p, mst in zip(ref.parameters(), masters):
                p.copy_(mst.to(torch.bfloat16))
        curve_ref.append(lr_)

    assert eng.launched_during_backward > 0
    # it trains ...
    assert curve_eng[-1] < 0.5 * curve_eng[0], (curve_eng[0], curve_eng[-1])
    # ... the first iteration sees identical parameters, so identical losses ...
    assert curve_eng[0] == curve_ref[0]
    # ... and the two curves stay together
    for t in range(STEPS):
        assert abs(curve_eng[t] - curve_ref[t]) <= 2e-2 * curve_ref[t], (t, curve_eng[t],
                                                                        curve_ref[t])
    eng.remove_hooks()


def test_engine_mixed_precision_step_and_training():
    """fp16 student with a dynamic loss scale starting at 2^24 (the first
    backward passes overflow fp16 and are skipped while the scale falls),
    clipping at 1.0.  Each iteration, the engine's step (overlapped bucket
    reductions that also sum squares, then zero_step_amp_reduced) must equal
    zero_step_amp run with the same bucket size on copies of the engine's own
    gradient replicas and state, bit for bit; and the model must train."""
    teacher = _mlp(123, torch.float32)
    student = _mlp(1, torch.float16)
    cfg = Z.AmpConfig(init_scale=2.0 ** 24, min_scale=1.0, window=20, hysteresis=1,
                      max_norm=1.0)
    hp = Z.AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01)
    eng = ZeroEngine(student.parameters(), N, mode="flat", align=16, op="avg", hparams=hp,
                     bucket_elems=20_000, overlap_comm=True, amp=cfg)
    plan = eng.plan

    def loss_of(model, x):
        with torch.no_grad():
            y = teacher(x)
        return (model(x.to(torch.float16)).float() - y).pow(2).mean()

    curve = []
    for t in range(STEPS):
        xs = [_micro_batch(q, t) for q in range(N)]
        le = 0.0
        for q in range(N):
            loss = loss_of(student, xs[q])
            eng.backward(loss, q)
            le += loss.item() / N
        curve.append(le)
        # the same step by zero_step_amp on copies of the replicas and state
        torch.cuda.current_stream().wait_stream(eng.reduction_stream)
        grads = [g.clone() for g in eng.grads]
        copies = {k: [x.clone() for x in getattr(eng, k)] for k in ("master", "m", "v")}
        state = eng.amp_state.clone()
        flat = eng.flat16.clone()
        gsh = [torch.empty_like(x) for x in eng.grad_shards]
        ws = torch.empty_like(eng._workspace)
        Z.zero_step_amp(plan, grads, "avg", gsh, copies["master"], copies["m"], copies["v"],
                        flat, None, hp, cfg, state, ws, bucket_elems=eng.bucket_elems)
        eng.step()
        torch.cuda.synchronize()
        assert torch.equal(state, eng.amp_state), t
        assert torch.equal(flat, eng.flat16), t
        for k in ("master", "m", "v"):
            for r in range(N):
                assert torch.equal(copies[k][r], getattr(eng, k)[r]), (t, k, r)
    st = eng.amp_status()
    assert st.skipped >= 1 and st.step == STEPS - st.skipped
    assert st.scale < 2.0 ** 24
    assert curve[-1] < 0.5 * curve[0], (curve[0], curve[-1])
    eng.remove_hooks()


@pytest.mark.parametrize("mode,overlap,bucket", [("round_robin", True, 20_000),
                                                 ("flat", False, 20_000),
                                                 ("flat", True, 0)])
def test_engine_mixed_precision_step_other_layouts(mode, overlap, bucket):
    """The engine's fp16 step equals zero_step_amp on copies of its replicas
    and state, bit for bit, for round-robin ownership, without overlap and
    with one bucket; 8 iterations from a scale of 2^20 (skips included)."""
    teacher = _mlp(321, torch.float32)
    student = _mlp(2, torch.float16)
    cfg = Z.AmpConfig(init_scale=2.0 ** 20, min_scale=1.0, window=3, hysteresis=2,
                      max_norm=0.5)
    hp = Z.AdamW(2e-3, 0.9, 0.99, 1e-8, 0.05)
    eng = ZeroEngine(student.parameters(), N, mode=mode, align=16, op="avg", hparams=hp,
                     bucket_elems=bucket, overlap_comm=overlap, amp=cfg)
    for t in range(8):
        xs = [_micro_batch(q, 100 + t) for q in range(N)]
        for q in range(N):
            with torch.no_grad():
                y = teacher(xs[q])
            eng.backward((student(xs[q].to(torch.float16)).float() - y).pow(2).mean(), q)
        if eng.reduction_stream is not None:
            torch.cuda.current_stream().wait_stream(eng.reduction_stream)
        grads = [g.clone() for g in eng.grads]
        copies = {k: [x.clone() for x in getattr(eng, k)] for k in ("master", "m", "v")}
        state = eng.amp_state.clone()
        flat = eng.flat16.clone()
        gsh = [torch.empty_like(x) for x in eng.grad_shards]
        ws = torch.empty_like(eng._workspace)
        Z.zero_step_amp(eng.plan, grads, "avg", gsh, copies["master"], copies["m"],
                        copies["v"], flat, None, hp, cfg, state, ws,
                        bucket_elems=eng.bucket_elems)
        eng.step()
        torch.cuda.synchronize()
        assert torch.equal(state, eng.amp_state), t
        assert torch.equal(flat.view(torch.int16), eng.flat16.view(torch.int16)), t
        for k in ("master", "m", "v"):
            for r in range(N):
                assert torch.equal(copies[k][r].view(torch.int32),
                                   getattr(eng, k)[r].view(torch.int32)), (t, k, r)
    assert eng.amp_status().step >= 1
    eng.remove_hooks()
