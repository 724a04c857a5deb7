"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small groups are compared element by element over whole buffers; the five
named parameter groups at full size are compared on sampled elements (seeded
random indices plus every shard, tensor, tile and bucket edge), which the
oracle recomputes one by one from the same inputs.  The launch configuration
is the one the benchmark uses (the library picks it; nothing here changes it).

Pass criteria: partition layout and gathered buffers bit-exact; fp32
master/m/v within 1e-6 relative error; 16-bit parameters within 1 ulp.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
from tests._harness import (Case, assert_16_close, assert_fp32_close, dt_code, f32, flat_len,
                            hp_oracle, op_code, owner_of, sample_indices, u16)
from zero_sharded_optimizer_flatten_gb300 import workloads as W
from zero_sharded_optimizer_flatten_gb300 import zero as Z

pytestmark = pytest.mark.gpu

HP = Z.AdamW(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@pytest.fixture(autouse=True)
def _cuda_cleanup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _run_full(w: W.Workload, steps: int, hp=HP, bucket=0, stream=None):
    c = Case(w)
    for t in range(1, steps + 1):
        g = c.grads(t)
        Z.zero_step(c.plan, g, w.op, c.master, c.m, c.v, c.full16, None, hp, t,
                    rank_mask=w.mask, bucket_elems=bucket, stream=stream)
        c.oracle_step(g, t, hp_oracle(hp))
    torch.cuda.synchronize()
    c.compare(f"{w.key} step {steps}")
    return c


# ----------------------------------------------------------------------------
# whole-buffer parity


def test_tiny_mlp_group_full():
    """The tiny-MLP group (1,053,706 params, fp16, N=4, A=16), 3 steps."""
    _run_full(W.WORKLOADS["tiny_mlp"], 3)


SMALL = [
    # numel, N, mode, A, dtype, op
    ((1000, 37, 4096, 3, 129, 0, 8191), 4, "flat", 16, "fp16", "avg"),
    ((1000, 37, 4096, 3, 129, 0, 8191), 4, "flat", 16, "bf16", "sum"),
    ((1000, 37, 4096, 3, 129, 0, 8191), 3, "flat", 2, "bf16", "avg"),   # unaligned shards
    ((1000, 37, 4096, 3, 129, 0, 8191), 5, "flat", 1, "fp16", "avg"),   # division by 5
    ((1000, 37, 4096, 3, 129, 0, 8191), 8, "flat", 8, "bf16", "avg"),
    ((1000, 37, 4096, 3, 129, 0, 8191), 1, "flat", 16, "fp16", "avg"),
    ((1000, 37, 4096, 3, 129, 0, 8191), 16, "flat", 16, "bf16", "avg"),  # generic-N path
    ((1000, 37, 4096, 3, 129, 0, 8191), 6, "round_robin", 1, "fp16", "sum"),
    ((1000, 37, 4096, 3, 129, 0, 8191), 9, "round_robin", 1, "bf16", "avg"),  # empty shards
    ((70001,), 7, "flat", 1, "fp16", "sum"),                             # one ragged tensor
    ((1,), 4, "flat", 16, "bf16", "avg"),                                # one element
    ((5, 3), 2, "round_robin", 1, "fp16", "avg"),
    ((1000, 37), 64, "flat", 4096, "bf16", "avg"),                       # largest A: 262,144
]


@pytest.mark.parametrize("numel,N,mode,A,dtype,op", SMALL)
def test_small_groups(numel, N, mode, A, dtype, op):
    w = W.small(numel, N, mode=mode, align=A, dtype=dtype, op=op, outlier_frac=0.01)
    _run_full(w, 3)


@pytest.mark.parametrize("hp", [Z.AdamW(lr=3e-2, beta1=0.8, beta2=0.95, eps=1e-6, weight_decay=0.1),
                                Z.AdamW(lr=1e-4, weight_decay=0.0)], ids=["aggressive", "wd0"])
def test_other_hyperparameters(hp):
    w = W.small((3000, 17, 555), 4, mode="flat", align=16, dtype="bf16", op="avg")
    _run_full(w, 4, hp=hp)


def _many_tensors(n=700, seed=3):
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(1, 3000, size=n))


def test_many_tensors_need_several_launches():
    """700 round-robin tensors of odd sizes over 3 ranks: every tensor is its
    own run, most split into head, quad body and tail jobs, so one call needs
    far more than the 192 jobs one launch carries; whole buffers and the
    16-bit shard outputs are compared with the oracle."""
    numel = _many_tensors()
    w = W.small(numel, 3, mode="round_robin", align=1, dtype="fp16", op="sum")
    plan = Z.zero_plan_partitions(list(numel), 3, "round_robin", 1)
    runs = sum(len(plan.segments(r)) for r in range(3))
    assert runs >= 700
    before = Z.zero_launch_count()
    c = _run_full(w, 2)
    assert Z.zero_launch_count() - before >= 2 * (runs // 192 + 1)
    s16 = [torch.empty(c.plan.shard_len(r), dtype=w.torch_dtype, device="cuda") for r in range(3)]
    g = c.grads(3)
    Z.zero_step(c.plan, g, "sum", c.master, c.m, c.v, c.full16, s16, HP, 3)
    o16 = [np.zeros(c.plan.shard_len(r), np.uint16) for r in range(3)]
    oracle.step(list(numel), 3, oracle.ROUND_ROBIN, 1, dt_code(w), oracle.SUM,
                [u16(x) for x in g], c.o_master, c.o_m, c.o_v, c.o_full, o16, hp_oracle(HP), 3)
    torch.cuda.synchronize()
    c.compare("many tensors step 3")
    for r in range(3):
        assert np.array_equal(u16(s16[r]), o16[r])


def test_unfused_calls_with_several_launches():
    """The unfused calls on the 700-tensor round-robin group, where each call
    needs several launches (every launch after a call's first starts early):
    zero_reduce_scatter bit for bit against the oracle's reduce-scatter,
    zero_adamw_shard_step with 16-bit shard outputs and zero_allgather against
    the oracle's step, over two steps."""
    numel = _many_tensors()
    w = W.small(numel, 3, mode="round_robin", align=1, dtype="fp16", op="sum")
    c = Case(w)
    gsh = [torch.empty(c.plan.shard_len(r), dtype=torch.float32, device="cuda") for r in range(3)]
    s16 = [torch.empty(c.plan.shard_len(r), dtype=w.torch_dtype, device="cuda") for r in range(3)]
    for t in (1, 2):
        g = c.grads(t)
        n0 = Z.zero_launch_count()
        Z.zero_reduce_scatter(c.plan, g, "sum", gsh)
        assert Z.zero_launch_count() - n0 >= 2
        torch.cuda.synchronize()
        orc = [np.zeros(c.plan.shard_len(r), np.float32) for r in range(3)]
        oracle.reduce_scatter(list(numel), 3, oracle.ROUND_ROBIN, 1, dt_code(w), oracle.SUM,
                              [u16(x) for x in g], orc)
        for r in range(3):
            assert np.array_equal(f32(gsh[r]).view(np.uint32), orc[r].view(np.uint32)), (t, r)
        n0 = Z.zero_launch_count()
        Z.zero_adamw_shard_step(c.plan, c.master, c.m, c.v, gsh, s16, HP, t)
        Z.zero_allgather(c.plan, s16, c.full16)
        assert Z.zero_launch_count() - n0 >= 4
        c.oracle_step(g, t, hp_oracle(HP))
        torch.cuda.synchronize()
        c.compare(f"unfused, several launches, step {t}")
        for r in range(3):
            seg = c.o_seg[r]
            o16 = np.zeros(c.plan.shard_len(r), np.uint16)
            for k, toff, foff, soff, ln in seg:
                o16[soff:soff + ln] = c.o_full[foff:foff + ln]
            assert_16_close(u16(s16[r]), o16, f"shard16[{r}] step {t}", dtype_code=dt_code(w))


@pytest.mark.parametrize("mode", ["flat", "round_robin"])
def test_groups_without_elements(mode):
    """Every tensor empty: the plan has no element, a step launches nothing
    and succeeds, and the oracle agrees that nothing changes."""
    numel = (0, 0, 0)
    plan = Z.zero_plan_partitions(list(numel), 4, mode, 16)
    assert (plan.phi, plan.padded) == (0, 0)
    assert all(plan.shard_len(r) == 0 for r in range(4))
    empty16 = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    empty32 = [torch.empty(0, dtype=torch.float32, device="cuda") for _ in range(4)]
    before = Z.zero_launch_count()
    Z.zero_step(plan, [empty16] * 4, "avg", empty32, empty32, empty32, empty16, None, HP, 1)
    Z.zero_sync()
    assert Z.zero_launch_count() == before


def test_large_step_count():
    """Bias-correction constants at t = 1000 (beta2^t far from 1)."""
    w = W.small((4096, 100), 2, mode="flat", align=16, dtype="fp16", op="avg")
    c = Case(w)
    for t in (999, 1000):
        g = c.grads(t)
        Z.zero_step(c.plan, g, w.op, c.master, c.m, c.v, c.full16, None, HP, t)
        c.oracle_step(g, t, hp_oracle(HP))
    torch.cuda.synchronize()
    c.compare("t=1000")


def test_non_default_stream():
    w = W.small((5000, 33), 4, mode="flat", align=16, dtype="bf16", op="avg")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c = _run_full(w, 2, stream=s)
    assert c is not None


def test_calls_from_several_host_threads():
    """The library keeps no shared mutable state between calls (plans are
    read-only; launch arguments are per call, events per thread, the error
    message thread-local): four host threads, each stepping its own group on
    its own stream (bucketed fused steps or the three unfused calls) and then
    failing one call on purpose, give the results of the same calls made one
    thread at a time, and each thread reads its own error message."""
    import threading
    w = W.small((30000, 37, 4096, 3, 129), 4, mode="flat", align=16, dtype="bf16", op="avg")

    def make():
        c = Case(w, with_oracle=False)
        c.gsh = [torch.empty(c.plan.shard_len(r), dtype=torch.float32, device="cuda")
                 for r in range(4)]
        c.s16 = [torch.empty(c.plan.shard_len(r), dtype=torch.bfloat16, device="cuda")
                 for r in range(4)]
        return c
    ref = [make() for _ in range(4)]
    got = [make() for _ in range(4)]
    grads = [ref[0].grads(t) for t in (1, 2, 3)]     # read-only, shared by every thread

    def run(c, k, stream, errors=None):
        for i, t in enumerate((1, 2, 3)):
            g = grads[i]
            if k % 2:
                Z.zero_step(c.plan, g, "avg", c.master, c.m, c.v, c.full16, None, HP, t,
                            bucket_elems=7000 + 1000 * k, stream=stream)
            else:
                Z.zero_reduce_scatter(c.plan, g, "avg", c.gsh, stream=stream)
                Z.zero_adamw_shard_step(c.plan, c.master, c.m, c.v, c.gsh, c.s16, HP, t,
                                        stream=stream)
                Z.zero_allgather(c.plan, c.s16, c.full16, stream=stream)
        if errors is not None:
            try:
                Z.zero_step(c.plan, grads[0], "avg", c.master, c.m, c.v, c.full16, None, HP,
                            -k, stream=stream)
            except Z.ZeroError as e:
                errors[k] = str(e)

    for k in range(4):
        run(ref[k], k, None)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(4)]
    errors = [None] * 4
    threads = [threading.Thread(target=run, args=(got[k], k, streams[k], errors))
               for k in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    for k in range(4):
        for r in range(4):
            assert torch.equal(got[k].master[r], ref[k].master[r]), (k, r)
            assert torch.equal(got[k].m[r], ref[k].m[r]), (k, r)
            assert torch.equal(got[k].v[r], ref[k].v[r]), (k, r)
        assert torch.equal(got[k].full16, ref[k].full16), k
        # each thread's message names its own bad step number
        assert errors[k] is not None and f"got {-k}" in errors[k], errors[k]


def test_init_shards_exact():
    w = W.small((1000, 37, 4096, 3), 3, mode="flat", align=2, dtype="bf16")
    c = Case(w)
    torch.cuda.synchronize()
    for r in range(w.n_ranks):
        assert np.array_equal(f32(c.master[r]).view(np.uint32), c.o_master[r].view(np.uint32))
        assert not f32(c.m[r]).any() and not f32(c.v[r]).any()


@pytest.mark.parametrize("bucket", [1, 7, 1000, 4096, 50_000])
def test_results_do_not_depend_on_buckets(bucket):
    w = W.small((30000, 37, 4096, 3, 129), 4, mode="flat", align=16, dtype="bf16", op="avg")
    ref = Case(w, with_oracle=False)
    got = Case(w, with_oracle=False)
    for t in (1, 2):
        g = ref.grads(t)
        Z.zero_step(ref.plan, g, "avg", ref.master, ref.m, ref.v, ref.full16, None, HP, t)
        Z.zero_step(got.plan, g, "avg", got.master, got.m, got.v, got.full16, None, HP, t,
                    bucket_elems=bucket)
    torch.cuda.synchronize()
    for r in range(4):
        assert torch.equal(ref.master[r], got.master[r])
        assert torch.equal(ref.m[r], got.m[r]) and torch.equal(ref.v[r], got.v[r])
    assert torch.equal(ref.full16, got.full16)


@pytest.mark.parametrize("mode,N,A", [("flat", 4, 16), ("round_robin", 4, 1), ("flat", 3, 2)])
def test_unfused_composition_is_bit_identical(mode, N, A):
    """reduce_scatter -> adamw_shard_step -> allgather == zero_step, and the
    pieces match the oracle's own unfused pieces."""
    w = W.small((20000, 37, 4096, 3, 129), N, mode=mode, align=A, dtype="fp16", op="avg")
    fused = Case(w, with_oracle=False)
    parts = Case(w, with_oracle=False)
    gsh = [torch.empty(parts.plan.shard_len(r), dtype=torch.float32, device="cuda")
           for r in range(N)]
    s16 = [torch.empty(parts.plan.shard_len(r), dtype=w.torch_dtype, device="cuda")
           for r in range(N)]
    for t in (1, 2):
        g = fused.grads(t)
        Z.zero_step(fused.plan, g, "avg", fused.master, fused.m, fused.v, fused.full16, None, HP, t)
        Z.zero_reduce_scatter(parts.plan, g, "avg", gsh)
        if t == 1:
            torch.cuda.synchronize()
            orc = [np.zeros(parts.plan.shard_len(r), np.float32) for r in range(N)]
            oracle.reduce_scatter(list(w.numel), N, oracle.FLAT if mode == "flat" else
                                  oracle.ROUND_ROBIN, A, dt_code(w), oracle.AVG,
                                  [u16(x) for x in g], orc)
            for r in range(N):
                assert np.array_equal(f32(gsh[r]).view(np.uint32), orc[r].view(np.uint32))
        Z.zero_adamw_shard_step(parts.plan, parts.master, parts.m, parts.v, gsh, s16, HP, t)
        Z.zero_allgather(parts.plan, s16, parts.full16)
    torch.cuda.synchronize()
    for r in range(N):
        assert torch.equal(fused.master[r], parts.master[r])
        assert torch.equal(fused.m[r], parts.m[r]) and torch.equal(fused.v[r], parts.v[r])
    assert torch.equal(fused.full16, parts.full16)


def test_rank_mask_touches_only_masked_ranks():
    w = W.small((5000, 37, 4096), 4, mode="flat", align=16, dtype="bf16", op="avg")
    c = Case(w)
    sentinel = float("nan")
    for r in (1, 3):
        c.master[r].fill_(sentinel)
        c.m[r].fill_(sentinel)
        c.v[r].fill_(sentinel)
    c.full16.fill_(7)
    before_full = u16(c.full16)
    g = c.grads(1)
    Z.zero_step(c.plan, g, "avg", c.master, c.m, c.v, c.full16, None, HP, 1, rank_mask=0b0101)
    c.oracle_step(g, 1, hp_oracle(HP), mask=0b0101)
    torch.cuda.synchronize()
    for r in (1, 3):
        assert torch.isnan(c.master[r]).all() and torch.isnan(c.v[r]).all()
    full = u16(c.full16)
    for r in (0, 2):
        off, ln = c.plan.shards[r]
        assert_16_close(full[off:off + ln], c.o_full[off:off + ln], f"full16 rank {r}")
        assert_fp32_close(f32(c.master[r]), c.o_master[r], f"master[{r}]")
    for r in (1, 3):
        off, ln = c.plan.shards[r]
        assert np.array_equal(full[off:off + ln], before_full[off:off + ln])


def test_zero3_shard_output():
    """out16_shard receives each rank's 16-bit shard, equal to its slot of
    the gathered buffer."""
    w = W.small((20000, 37, 4096, 3, 129), 4, mode="flat", align=16, dtype="bf16", op="avg")
    c = Case(w)
    s16 = [torch.empty(c.plan.shard_len(r), dtype=w.torch_dtype, device="cuda") for r in range(4)]
    g = c.grads(1)
    Z.zero_step(c.plan, g, "avg", c.master, c.m, c.v, c.full16, s16, HP, 1)
    c.oracle_step(g, 1, hp_oracle(HP))
    torch.cuda.synchronize()
    c.compare("zero3")
    for r in range(4):
        off, ln = c.plan.shards[r]
        assert torch.equal(s16[r], c.full16[off:off + ln])


# ----------------------------------------------------------------------------
# full-size groups, sampled parity


def _sampled(w: W.Workload, steps: int, hp=HP, n_random=20000, extra=()):
    """Run the CUDA step at full size and check sampled elements against the
    oracle recomputing those elements one by one from the same inputs."""
    extra = list(extra)
    if w.bucket_elems:
        extra += list(range(0, flat_len(w), w.bucket_elems))
    F = sample_indices(w, n_random=n_random, extra=extra)
    rank, shard = owner_of(w, F)
    keep = np.array([(w.mask >> int(r)) & 1 for r in rank], bool) & (rank >= 0)
    F, rank, shard = F[keep], rank[keep], shard[keep]
    Ft = torch.from_numpy(F).cuda()
    c = Case(w, with_oracle=False)
    ext = c.plan.flat_extent(w.mask)
    dt, op = dt_code(w), op_code(w)
    om = oracle.to_f32(u16(c.p16[Ft]), dt)
    mm, vv = np.zeros_like(om), np.zeros_like(om)
    out = np.zeros(F.size, np.uint16)
    for t in range(1, steps + 1):
        g = [W.grads16(w, t, q, "cuda", 0, ext) for q in range(w.n_ranks)]
        gs = np.stack([u16(x[Ft]) for x in g])
        Z.zero_step(c.plan, g, w.op, c.master, c.m, c.v, c.full16[:ext], None, hp, t,
                    rank_mask=w.mask, bucket_elems=w.bucket_elems)
        oracle.update_elements(gs, om, mm, vv, dt, op, hp_oracle(hp), t, out16=out)
        del g
    torch.cuda.synchronize()
    got_p = np.empty(F.size, np.float32)
    got_m = np.empty(F.size, np.float32)
    got_v = np.empty(F.size, np.float32)
    for r in np.unique(rank):
        sel = rank == r
        it = torch.from_numpy(shard[sel]).cuda()
        got_p[sel] = f32(c.master[r][it])
        got_m[sel] = f32(c.m[r][it])
        got_v[sel] = f32(c.v[r][it])
    assert_fp32_close(got_p, om, f"{w.key} master")
    assert_fp32_close(got_m, mm, f"{w.key} m")
    assert_fp32_close(got_v, vv, f"{w.key} v")
    assert_16_close(u16(c.full16[Ft]), out, f"{w.key} full16")
    return F.size


# Flat and shard indices past 2^31 and 2^32: every offset the kernels form is
# 64-bit.  Round-robin groups put a small tensor behind a huge one, so one
# rank's elements sit at large flat offsets (and, in the first case, rank 0's
# last tensor at a shard offset past 2^31).  Odd lengths put element-wise
# jobs there as well as quad jobs.
LARGE_INDEX = [
    # numel, rank mask, device bytes needed (replicas, parameters, gathered buffer, state)
    ((2_200_000_000, 6001, 4003), 0b11, 46 << 30),
    ((4_300_000_000, 6001), 0b10, 36 << 30),
]


@pytest.mark.parametrize("numel,mask,need", LARGE_INDEX, ids=["past_2^31", "past_2^32"])
def test_indices_past_32_bits_sampled(numel, mask, need):
    free, _ = torch.cuda.mem_get_info()
    if free < need + (4 << 30):
        pytest.skip(f"needs {need >> 30} GiB of free device memory")
    w = W.small(numel, 2, mode="round_robin", align=1, dtype="bf16", op="sum", rank_mask=mask)
    starts = np.concatenate([[0], np.cumsum(np.asarray(numel, np.int64))])
    extra = list(range(int(starts[1]), int(starts[-1])))        # every small-tensor element
    for b in (1 << 31, 1 << 32):
        extra += [x for x in range(b - 4100, b + 4100) if x < starts[-1]]
    assert _sampled(w, 2, n_random=4000, extra=extra) >= 6001
    gc.collect()
    torch.cuda.empty_cache()


def test_bert_base_full_size_sampled():
    assert _sampled(W.WORKLOADS["bert_base"], 10) > 20000


def test_toy_model_round_robin_full_size_sampled():
    assert _sampled(W.WORKLOADS["toy_rr"], 3) > 20000


def test_llama7b_rank0_shard_full_size_sampled():
    """Rank 0's 842M-element shard, 8 bf16 gradient slices, 50M-element
    buckets (the gradient buffers hold only rank 0's flat range)."""
    assert _sampled(W.WORKLOADS["llama7b_rank0"], 3, n_random=8000) > 8000


def test_llama7b_rank0_shard_whole_buckets():
    """Whole 50M-element buckets of rank 0's shard (the first, the last and two
    seeded ones) over the three steps, every element against the oracle: the
    step is element-wise, so whole buckets check everything a bucket launch
    writes, including its tile and launch edges."""
    w = W.WORKLOADS["llama7b_rank0"]
    B = w.bucket_elems
    seg = oracle.segments(list(w.numel), w.n_ranks, oracle.FLAT, w.align, 0)
    assert (seg[:, 2] == seg[:, 3]).all()           # rank 0: shard index = flat index
    S = int(seg[:, 4].sum())
    nb = -(-S // B)
    rng = np.random.default_rng(7)
    picks = sorted({0, nb - 1, *[int(x) for x in rng.choice(np.arange(1, nb - 1), 2, False)]})
    c = Case(w, with_oracle=False)
    ext = c.plan.flat_extent(w.mask)
    assert ext == S
    dt, op, hp = dt_code(w), op_code(w), hp_oracle(HP)
    ranges = [(b * B, min(S, (b + 1) * B)) for b in picks]
    state = []
    for lo, hi in ranges:
        om = oracle.to_f32(u16(c.p16[lo:hi]), dt)
        state.append([om, np.zeros_like(om), np.zeros_like(om), np.zeros(hi - lo, np.uint16)])
    for t in range(1, 4):
        g = [W.grads16(w, t, q, "cuda", 0, ext) for q in range(w.n_ranks)]
        Z.zero_step(c.plan, g, w.op, c.master, c.m, c.v, c.full16[:ext], None, HP, t,
                    rank_mask=w.mask, bucket_elems=B)
        for (lo, hi), (om, mm, vv, out) in zip(ranges, state):
            gs = np.stack([u16(x[lo:hi]) for x in g])
            oracle.update_elements(gs, om, mm, vv, dt, op, hp, t, out16=out)
        del g
    torch.cuda.synchronize()
    for b, (lo, hi), (om, mm, vv, out) in zip(picks, ranges, state):
        what = f"bucket {b} [{lo}, {hi})"
        assert_fp32_close(f32(c.master[0][lo:hi]), om, what + " master")
        assert_fp32_close(f32(c.m[0][lo:hi]), mm, what + " m")
        assert_fp32_close(f32(c.v[0][lo:hi]), vv, what + " v")
        assert_16_close(u16(c.full16[lo:hi]), out, what + " full16", dtype_code=dt)


@pytest.mark.parametrize("key", ["llama13b_layer", "llama13b_full_layer"])
def test_llama13b_zero3_layer_pass_sampled(key):
    """Two layers of the ZeRO-3 stream (the 3 MLP matrices, or the whole
    decoder layer): all-gather 8 bf16 shards into the layer buffer
    (bit-exact), then the fused step writing each rank's shard."""
    w = W.WORKLOADS[key]
    plan = Z.zero_plan_partitions(list(w.numel), w.n_ranks, w.mode, w.align)
    L = flat_len(w)
    S = plan.shard_len(0)
    layer_buf = torch.empty(L, dtype=w.torch_dtype, device="cuda")
    F = sample_indices(w, n_random=8000)
    rank, shard = owner_of(w, F)
    Ft = torch.from_numpy(F).cuda()
    dt, op = dt_code(w), op_code(w)
    for layer in range(2):
        p16 = W.params16(w, "cuda", L, layer=layer)
        shards = [p16[r * S:(r + 1) * S].clone() for r in range(w.n_ranks)]
        master = [torch.empty(S, dtype=torch.float32, device="cuda") for _ in range(w.n_ranks)]
        m = [torch.empty_like(x) for x in master]
        v = [torch.empty_like(x) for x in master]
        Z.zero_init_shards(plan, p16, master, m, v)
        Z.zero_allgather(plan, shards, layer_buf)
        torch.cuda.synchronize()
        assert torch.equal(layer_buf, p16)
        om = oracle.to_f32(u16(p16[Ft]), dt)
        mm, vv = np.zeros_like(om), np.zeros_like(om)
        out = np.zeros(F.size, np.uint16)
        g = [W.grads16(w, 1, q, "cuda", 0, L, layer=layer) for q in range(w.n_ranks)]
        gs = np.stack([u16(x[Ft]) for x in g])
        Z.zero_step(plan, g, "avg", master, m, v, None, shards, HP, 1)
        oracle.update_elements(gs, om, mm, vv, dt, op, hp_oracle(HP), 1, out16=out)
        torch.cuda.synchronize()
        for r in range(w.n_ranks):
            sel = rank == r
            it = torch.from_numpy(shard[sel]).cuda()
            assert_fp32_close(f32(master[r][it]), om[sel], f"layer {layer} master[{r}]")
            assert_fp32_close(f32(m[r][it]), mm[sel], f"layer {layer} m[{r}]")
            assert_fp32_close(f32(v[r][it]), vv[sel], f"layer {layer} v[{r}]")
            assert_16_close(u16(shards[r][it]), out[sel], f"layer {layer} shard16[{r}]")
        # the next gather reproduces the updated shards in the layer buffer
        Z.zero_allgather(plan, shards, layer_buf)
        torch.cuda.synchronize()
        assert torch.equal(layer_buf, torch.cat(shards))
        del g, shards, master, m, v, p16


@pytest.mark.parametrize("mode,N,dtype", [("flat", 8, "bf16"), ("round_robin", 4, "fp16")])
def test_host_buffers_through_the_link(mode, N, dtype):
    """Gradient replicas in pinned host memory and the gathered parameters
    written to pinned host memory: bit-identical to device buffers."""
    w = W.small((30000, 37, 4096, 3, 129), N, mode=mode, align=16, dtype=dtype, op="avg")
    dev_case = Case(w, with_oracle=False)
    host_case = Case(w, with_oracle=False)
    host_full = torch.zeros(host_case.L, dtype=w.torch_dtype, pin_memory=True)
    for t in (1, 2):
        g = dev_case.grads(t)
        hg = [x.cpu().pin_memory() for x in g]
        Z.zero_step(dev_case.plan, g, "avg", dev_case.master, dev_case.m, dev_case.v,
                    dev_case.full16, None, HP, t)
        Z.zero_step(host_case.plan, hg, "avg", host_case.master, host_case.m, host_case.v,
                    host_full, None, HP, t)
        torch.cuda.synchronize()
    for r in range(N):
        assert torch.equal(dev_case.master[r], host_case.master[r])
        assert torch.equal(dev_case.v[r], host_case.v[r])
    assert torch.equal(dev_case.full16.cpu(), host_full)


def test_optimizer_state_in_host_memory():
    """ZeRO-Offload over the host link: fp32 master/m/v in pinned host memory,
    gradients and parameters in HBM; bit-identical to device-resident state,
    through init, the fused step and the unfused pieces."""
    w = W.small((30000, 37, 4096, 3, 129), 4, mode="flat", align=16, dtype="bf16", op="avg")
    dev_case = Case(w)
    plan = dev_case.plan
    S = [plan.shard_len(r) for r in range(4)]
    hm = [torch.empty(n, dtype=torch.float32, pin_memory=True) for n in S]
    hmm = [torch.empty(n, dtype=torch.float32, pin_memory=True) for n in S]
    hv = [torch.empty(n, dtype=torch.float32, pin_memory=True) for n in S]
    full = torch.zeros_like(dev_case.full16)
    Z.zero_init_shards(plan, dev_case.p16, hm, hmm, hv)
    for t in (1, 2):
        g = dev_case.grads(t)
        Z.zero_step(plan, g, "avg", dev_case.master, dev_case.m, dev_case.v, dev_case.full16, None,
                    HP, t)
        Z.zero_step(plan, g, "avg", hm, hmm, hv, full, None, HP, t)
        dev_case.oracle_step(g, t, hp_oracle(HP))
    torch.cuda.synchronize()
    for r in range(4):
        assert torch.equal(dev_case.master[r].cpu(), hm[r])
        assert torch.equal(dev_case.m[r].cpu(), hmm[r]) and torch.equal(dev_case.v[r].cpu(), hv[r])
        # the host-resident state against the oracle
        assert_fp32_close(hm[r].numpy(), dev_case.o_master[r], f"host master[{r}]")
        assert_fp32_close(hmm[r].numpy(), dev_case.o_m[r], f"host m[{r}]")
        assert_fp32_close(hv[r].numpy(), dev_case.o_v[r], f"host v[{r}]")
    assert torch.equal(dev_case.full16, full)
    assert_16_close(u16(full), dev_case.o_full, "full16", dtype_code=dt_code(w))


def test_cpu_optimizer_offload_pipeline():
    """ZeRO-Offload with the CPU optimizer: the GPU reduce-scatters into pinned
    host fp32 shards, host threads run AdamW on host-resident state, the GPU
    all-gathers the host 16-bit shards.  Bit-identical to the fused step."""
    w = W.small((30000, 37, 4096, 3, 129), 4, mode="flat", align=16, dtype="bf16", op="avg")
    dev_case = Case(w)
    plan = dev_case.plan
    S = [plan.shard_len(r) for r in range(4)]
    pin = lambda n, dt: torch.zeros(n, dtype=dt, pin_memory=True)  # noqa: E731
    hm = [dev_case.master[r].cpu().pin_memory() for r in range(4)]
    hmm = [pin(n, torch.float32) for n in S]
    hv = [pin(n, torch.float32) for n in S]
    hg = [pin(n, torch.float32) for n in S]
    h16 = [pin(n, w.torch_dtype) for n in S]
    full = torch.zeros_like(dev_case.full16)
    for t in (1, 2, 3):
        g = dev_case.grads(t)
        Z.zero_step(plan, g, "avg", dev_case.master, dev_case.m, dev_case.v, dev_case.full16, None,
                    HP, t)
        Z.zero_reduce_scatter(plan, g, "avg", hg)
        Z.zero_sync()
        Z.zero_cpu_adamw_shard_step(plan, hm, hmm, hv, hg, h16, HP, t, Z.ZERO_BF16)
        Z.zero_allgather(plan, h16, full)
        dev_case.oracle_step(g, t, hp_oracle(HP))
    torch.cuda.synchronize()
    for r in range(4):
        assert torch.equal(dev_case.master[r].cpu(), hm[r])
        assert torch.equal(dev_case.v[r].cpu(), hv[r])
        # the host optimizer's state and 16-bit shards against the oracle
        assert_fp32_close(hm[r].numpy(), dev_case.o_master[r], f"host master[{r}]")
        assert_fp32_close(hmm[r].numpy(), dev_case.o_m[r], f"host m[{r}]")
        assert_fp32_close(hv[r].numpy(), dev_case.o_v[r], f"host v[{r}]")
        off = int(dev_case.o_seg[r][0, 2])          # flat offset of the shard (oracle plan)
        assert_16_close(u16(h16[r]), dev_case.o_full[off:off + S[r]], f"host shard16[{r}]",
                        dtype_code=dt_code(w))
    assert torch.equal(dev_case.full16, full)
    assert_16_close(u16(full), dev_case.o_full, "full16", dtype_code=dt_code(w))



def _host_offload_state(c: Case):
    """Host copies of a fresh case's shards: master in pinned memory, m/v in
    pageable host memory (allowed), pinned fp32 gradient and 16-bit shards."""
    S = [c.plan.shard_len(r) if (c.w.mask >> r) & 1 else 0 for r in range(c.w.n_ranks)]
    pin = lambda n, dt: torch.zeros(n, dtype=dt, pin_memory=True)  # noqa: E731
    hm = [c.master[r].cpu().pin_memory() for r in range(c.w.n_ranks)]
    hmm = [torch.zeros(n, dtype=torch.float32) for n in S]
    hv = [torch.zeros(n, dtype=torch.float32) for n in S]
    hg = [pin(n, torch.float32) for n in S]
    h16 = [pin(n, c.w.torch_dtype) for n in S]
    return hm, hmm, hv, hg, h16


@pytest.mark.parametrize("numel,N,mode,dtype,op,mask,chunk,threads", [
    ((30000, 37, 4096, 3, 129), 4, "flat", "bf16", "avg", None, None, 0),
    ((30000, 37, 4096, 3, 129), 4, "flat", "bf16", "avg", None, 0, 3),
    ((30000, 37, 4096, 3, 129), 4, "flat", "bf16", "avg", None, 1000, 5),
    ((30000, 37, 4096, 3, 129), 4, "flat", "fp16", "sum", 0b1010, 2999, 2),
    ((5000, 7, 12000, 1, 333, 9000), 3, "round_robin", "fp16", "sum", None, 4097, 4),
    ((20000, 17), 5, "flat", "bf16", "avg", None, 13, 1),
])
def test_pipelined_offload_step(numel, N, mode, dtype, op, mask, chunk, threads):
    """zero_offload_step (device reduce of chunk k+1 while host threads update
    chunk k, gather of each finished chunk) against the oracle, and bit for bit
    against the serial offload calls, over chunk sizes that cut tensors,
    shards and tiles anywhere, one chunk, rank masks and both layouts."""
    w = W.small(numel, N, mode=mode, align=16, dtype=dtype, op=op, rank_mask=mask)
    c = Case(w)
    plan = c.plan
    hm, hmm, hv, hg, h16 = _host_offload_state(c)
    sm, smm, sv, sg, s16 = _host_offload_state(c)
    full = torch.zeros_like(c.full16)
    sfull = torch.zeros_like(c.full16)
    dt = Z.ZERO_BF16 if dtype == "bf16" else Z.ZERO_FP16
    for t in (1, 2, 3):
        g = c.grads(t)
        Z.zero_offload_step(plan, g, op, hg, hm, hmm, hv, h16, full, HP, t, rank_mask=w.mask,
                            chunk_elems=chunk, n_threads=threads)
        Z.zero_reduce_scatter(plan, g, op, sg, rank_mask=w.mask)
        Z.zero_sync()
        Z.zero_cpu_adamw_shard_step(plan, sm, smm, sv, sg, s16, HP, t, dt, rank_mask=w.mask)
        Z.zero_allgather(plan, s16, sfull, rank_mask=w.mask)
        c.oracle_step(g, t, hp_oracle(HP))
    torch.cuda.synchronize()
    for r in range(N):
        if not (w.mask >> r) & 1:
            continue
        for got, ser, ref, what in ((hm, sm, c.o_master, "master"), (hmm, smm, c.o_m, "m"),
                                    (hv, sv, c.o_v, "v")):
            assert torch.equal(got[r], ser[r]), f"{what}[{r}] differs from the serial calls"
            assert_fp32_close(got[r].numpy(), ref[r], f"offload {what}[{r}]")
        assert torch.equal(h16[r], s16[r])
        seg = c.o_seg[r]
        want = np.concatenate([c.o_full[f:f + n] for _, _, f, _, n in seg]) if len(seg) else \
            np.zeros(0, np.uint16)
        assert_16_close(u16(h16[r]), want, f"offload shard16[{r}]", dtype_code=dt_code(w))
    assert torch.equal(full, sfull)
    owned = np.zeros(plan.padded, bool)
    for r in range(N):
        if (w.mask >> r) & 1:
            for _, _, f, _, n in c.o_seg[r]:
                owned[f:f + n] = True
    assert_16_close(u16(full)[owned], c.o_full[owned], "offload full16", dtype_code=dt_code(w))
    assert not u16(full)[~owned].any(), "an unmasked rank's elements were written"


def test_pipelined_offload_step_edge_cases():
    """A group without elements (nothing launched), no gathered buffer (the
    host 16-bit shards are still written) and a chunk larger than the flat
    buffer (one chunk)."""
    plan = Z.zero_plan_partitions([0, 0], 2, "flat", 16)
    empty16 = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    null = [0, 0]          # empty shards need no buffer (NULL addresses)
    before = Z.zero_launch_count()
    Z.zero_offload_step(plan, [empty16] * 2, "avg", null, null, null, null, null, empty16, HP, 1,
                        dtype=Z.ZERO_BF16)
    assert Z.zero_launch_count() == before
    w = W.small((30000, 37), 2, mode="flat", align=16, dtype="bf16", op="avg")
    c = Case(w)
    hm, hmm, hv, hg, h16 = _host_offload_state(c)
    for t in (1, 2):
        g = c.grads(t)
        Z.zero_offload_step(c.plan, g, "avg", hg, hm, hmm, hv, h16, None, HP, t,
                            chunk_elems=10 ** 9)
        Z.zero_step(c.plan, g, "avg", c.master, c.m, c.v, c.full16, None, HP, t)
    torch.cuda.synchronize()
    for r in range(2):
        assert torch.equal(hm[r], c.master[r].cpu())
        off = c.plan.shards[r][0]
        assert torch.equal(h16[r], c.full16[off:off + c.plan.shard_len(r)].cpu())

@pytest.mark.parametrize("chunk", [None, 0, 777])
def test_offload_step_from_reduced_shards(chunk):
    """grads=None: the gradient shards were reduced before the call (here by
    zero_reduce_scatter on the same stream, with no synchronisation in
    between); the step waits for that work, updates on the host and
    gathers, bit for bit like the serial calls."""
    w = W.small((30000, 37, 4096), 4, mode="round_robin", align=16, dtype="fp16", op="sum")
    c = Case(w, with_oracle=False)
    hm, hmm, hv, hg, h16 = _host_offload_state(c)
    sm, smm, sv, sg, s16 = _host_offload_state(c)
    full = torch.zeros_like(c.full16)
    sfull = torch.zeros_like(c.full16)
    for t in (1, 2):
        g = c.grads(t)
        Z.zero_reduce_scatter(c.plan, g, "sum", hg)
        Z.zero_offload_step(c.plan, None, "sum", hg, hm, hmm, hv, h16, full, HP, t,
                            chunk_elems=chunk, n_threads=3)
        Z.zero_reduce_scatter(c.plan, g, "sum", sg)
        Z.zero_sync()
        Z.zero_cpu_adamw_shard_step(c.plan, sm, smm, sv, sg, s16, HP, t, Z.ZERO_FP16)
        Z.zero_allgather(c.plan, s16, sfull)
    torch.cuda.synchronize()
    for r in range(4):
        assert torch.equal(hm[r], sm[r]) and torch.equal(hv[r], sv[r])
        assert torch.equal(h16[r], s16[r])
    assert torch.equal(full, sfull)

def test_pipelined_offload_step_rejects_bad_arguments_without_launching():
    w = W.small((30000, 37), 2, mode="flat", align=16, dtype="bf16", op="avg")
    c = Case(w, with_oracle=False)
    hm, hmm, hv, hg, h16 = _host_offload_state(c)
    g = c.grads(1)
    before = Z.zero_launch_count()
    # raw addresses pass the binding's own checks and reach the library's
    pageable = [torch.zeros(c.plan.shard_len(r), dtype=torch.float32) for r in range(2)]
    with pytest.raises(Z.ZeroError, match="pinned"):
        Z.zero_offload_step(c.plan, g, "avg", [t.data_ptr() for t in pageable], hm, hmm, hv,
                            h16, c.full16, HP, 1)
    with pytest.raises(Z.ZeroError, match="device memory"):
        Z.zero_offload_step(c.plan, g, "avg", hg, [t.data_ptr() for t in c.master], hmm, hv,
                            h16, c.full16, HP, 1)
    with pytest.raises(Z.ZeroError, match="chunks"):
        Z.zero_offload_step(c.plan, g, "avg", hg, hm, hmm, hv, h16, c.full16, HP, 1,
                            chunk_elems=7)
    with pytest.raises(Z.ZeroError, match="must be >= 1"):
        Z.zero_offload_step(c.plan, g, "avg", hg, hm, hmm, hv, h16, c.full16, HP, 0)
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    x = torch.zeros(4, device="cuda")
    with torch.cuda.stream(side):
        graph.capture_begin()
        x.add_(1)
        try:
            with pytest.raises(Z.ZeroError, match="captured"):
                Z.zero_offload_step(c.plan, g, "avg", hg, hm, hmm, hv, h16, c.full16, HP, 1,
                                    stream=side)
        finally:
            graph.capture_end()
    torch.cuda.synchronize()
    assert Z.zero_launch_count() == before
    assert not any(t.any() for t in h16) and not any(t.any() for t in hg)

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_non_finite_gradients_propagate_like_the_oracle(dtype):
    """+inf, -inf and NaN in one replica: the plain step propagates them as
    IEEE arithmetic does, on the same elements as the oracle (the update
    with overflow checks is zero_step_amp)."""
    w = W.small((4096, 37), 4, mode="flat", align=16, dtype=dtype, op="avg")
    c = Case(w)
    g = c.grads(1)
    g[2][10] = float("inf")
    g[2][11] = float("-inf")
    g[1][12] = float("nan")
    g[0][13] = float("inf")
    g[3][13] = float("-inf")          # inf + -inf -> NaN
    Z.zero_step(c.plan, g, "avg", c.master, c.m, c.v, c.full16, None, HP, 1)
    c.oracle_step(g, 1, hp_oracle(HP))
    torch.cuda.synchronize()
    c.compare("non-finite")
    assert np.isnan(f32(c.master[0])[10:14]).all()
