"""Parity of the mixed-precision step (loss scaling, overflow skip, global-norm
clipping) between the CUDA path and the oracle.

The squared norm is summed differently on the two sides: the oracle adds the
binary32 squares one after another in binary64; the CUDA path adds them per
tile and then across tiles in pairs of binary32 numbers (about 48
significant bits).  Both carry far more bits than the squares, so the norms
agree to 1e-10 relative (NORM_RTOL); the clip coefficient, rounded once to
binary32, may still differ in its last bit when clipping is active.  The
state's integer fields, the loss scale and every skip decision must agree
exactly, the coefficient to 1 ulp, and the buffers to the usual bar.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
from tests._harness import (Case, assert_16_close, assert_fp32_close, dt_code, f32, hp_oracle,
                            mode_code, op_code, owner_of, sample_indices, u16)
from zero_sharded_optimizer_flatten_gb300 import workloads as W
from zero_sharded_optimizer_flatten_gb300 import zero as Z

pytestmark = pytest.mark.gpu

HP = Z.AdamW()
NORM_RTOL = 1e-10


@pytest.fixture(autouse=True)
def _cuda_cleanup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _ocfg(c: Z.AmpConfig):
    return oracle.amp_config(c.init_scale, c.min_scale, c.window, c.hysteresis, c.max_norm)


class AmpCase(Case):
    def __init__(self, w, cfg: Z.AmpConfig, bucket=0, with_oracle=True):
        super().__init__(w, with_oracle=with_oracle)
        self.cfg, self.bucket = cfg, bucket
        self.gsh = [torch.empty(self.plan.shard_len(r) if (w.mask >> r) & 1 else 0,
                                dtype=torch.float32, device="cuda") for r in range(w.n_ranks)]
        self.state = Z.amp_state_tensor()
        Z.zero_amp_init(self.state, cfg)
        nbytes = Z.zero_amp_workspace_bytes(self.plan, w.mask, bucket)
        self.ws = torch.empty(max(16, nbytes), dtype=torch.uint8, device="cuda")
        self.ost = oracle.amp_init(_ocfg(cfg)) if with_oracle else None

    def grads_scaled(self, t, scale):
        return [W.grads16(self.w, t, q, "cuda", 0, self.L, scale=scale)
                for q in range(self.w.n_ranks)]

    def gpu_step(self, g):
        Z.zero_step_amp(self.plan, g, self.w.op, self.gsh, self.master, self.m, self.v,
                        self.full16, None, HP, self.cfg, self.state, self.ws,
                        rank_mask=self.w.mask, bucket_elems=self.bucket)

    def oracle_step_amp(self, g):
        w = self.w
        oracle.step_amp(list(w.numel), w.n_ranks, mode_code(w), w.align, dt_code(w), op_code(w),
                        [u16(x) for x in g], self.o_master, self.o_m, self.o_v, self.o_full, None,
                        hp_oracle(HP), _ocfg(self.cfg), self.ost, w.mask)

    def compare_state(self, what):
        s = Z.read_amp_state(self.state)
        o = self.ost
        assert (s.step, s.skipped, s.good_steps, s.hysteresis_left, s.overflow) == \
            (o.step, o.skipped, o.good_steps, o.hysteresis_left, o.overflow), what
        assert s.scale == o.scale, what
        if o.overflow:
            assert not np.isfinite(s.norm), what
        else:
            assert abs(s.norm - o.norm) <= NORM_RTOL * abs(o.norm), (what, s.norm, o.norm)
            d = abs(int(np.float32(s.coef).view(np.int32)) - int(np.float32(o.coef).view(np.int32)))
            assert d <= 1, (what, s.coef, o.coef)
        return s


CASES = [
    # numel, N, mode, A, dtype, op, cfg
    ((1000, 37, 4096, 3, 129), 4, "flat", 16, "fp16", "avg",
     Z.AmpConfig(init_scale=1024.0, window=3, hysteresis=2, max_norm=0.0)),
    ((1000, 37, 4096, 3, 129), 4, "flat", 16, "fp16", "sum",
     Z.AmpConfig(init_scale=256.0, window=1000, hysteresis=1, max_norm=0.05)),
    ((1000, 37, 4096, 3, 129), 3, "round_robin", 1, "bf16", "avg",
     Z.AmpConfig(init_scale=1.0, window=0, hysteresis=1, max_norm=0.01)),
    ((70001,), 8, "flat", 2, "bf16", "avg",
     Z.AmpConfig(init_scale=8.0, window=2, hysteresis=1, max_norm=0.02)),
]


@pytest.mark.parametrize("numel,N,mode,A,dtype,op,cfg", CASES)
def test_amp_small_groups(numel, N, mode, A, dtype, op, cfg):
    w = W.small(numel, N, mode=mode, align=A, dtype=dtype, op=op, outlier_frac=0.01)
    c = AmpCase(w, cfg)
    for t in range(1, 5):
        g = c.grads_scaled(t, c.ost.scale)
        c.gpu_step(g)
        c.oracle_step_amp(g)
        torch.cuda.synchronize()
        c.compare_state(f"step {t}")
        c.compare(f"amp step {t}")


def test_amp_overflow_trajectory():
    """A loss scale of 2^20 overflows fp16 gradients: the steps are skipped and
    the scale falls until the gradients fit, then updates resume."""
    w = W.small((3000, 129, 4096), 4, mode="flat", align=16, dtype="fp16", op="avg")
    cfg = Z.AmpConfig(init_scale=2.0 ** 20, min_scale=1.0, window=4, hysteresis=2)
    c = AmpCase(w, cfg)
    seen_skip = seen_step = False
    for t in range(1, 13):
        g = c.grads_scaled(t, c.ost.scale)
        c.gpu_step(g)
        c.oracle_step_amp(g)
        torch.cuda.synchronize()
        s = c.compare_state(f"call {t}")
        seen_skip |= bool(s.overflow)
        seen_step |= not s.overflow
        c.compare(f"call {t}")
    assert seen_skip and seen_step


def test_amp_skip_leaves_buffers_untouched():
    w = W.small((5000, 33), 2, mode="flat", align=16, dtype="fp16", op="sum")
    c = AmpCase(w, Z.AmpConfig(init_scale=4.0, hysteresis=1))
    g = c.grads_scaled(1, 4.0)
    c.gpu_step(g)
    torch.cuda.synchronize()
    before = [x.clone() for x in c.master + c.m + c.v] + [c.full16.clone()]
    g = c.grads_scaled(2, 4.0)
    g[1][777] = float("nan")
    c.gpu_step(g)
    torch.cuda.synchronize()
    s = Z.read_amp_state(c.state)
    assert s.overflow == 1 and s.step == 1 and s.skipped == 1 and s.scale == 2.0
    after = [x for x in c.master + c.m + c.v] + [c.full16]
    for a, b in zip(before, after):
        assert torch.equal(a, b)


def test_amp_unit_scale_is_the_fused_step():
    """S = 1 and no clipping: bit-identical to zero_step."""
    w = W.small((20000, 37, 4096, 3, 129), 4, mode="flat", align=16, dtype="bf16", op="avg")
    c = AmpCase(w, Z.AmpConfig(init_scale=1.0, window=0, hysteresis=1), with_oracle=False)
    ref = Case(w, with_oracle=False)
    for t in (1, 2, 3):
        g = c.grads_scaled(t, 1.0)
        c.gpu_step(g)
        Z.zero_step(ref.plan, g, "avg", ref.master, ref.m, ref.v, ref.full16, None, HP, t)
    torch.cuda.synchronize()
    for r in range(4):
        assert torch.equal(c.master[r], ref.master[r]) and torch.equal(c.v[r], ref.v[r])
    assert torch.equal(c.full16, ref.full16)


@pytest.mark.parametrize("bucket", [1000, 4096])
def test_amp_buckets(bucket):
    w = W.small((30000, 37, 4096), 4, mode="flat", align=16, dtype="bf16", op="avg")
    cfg = Z.AmpConfig(init_scale=1.0, window=0, hysteresis=1, max_norm=0.0)
    a = AmpCase(w, cfg, with_oracle=False)
    b = AmpCase(w, cfg, bucket=bucket, with_oracle=False)
    for t in (1, 2):
        g = a.grads_scaled(t, 1.0)
        a.gpu_step(g)
        b.gpu_step(g)
    torch.cuda.synchronize()
    for r in range(4):
        assert torch.equal(a.master[r], b.master[r])
    sa, sb = Z.read_amp_state(a.state), Z.read_amp_state(b.state)
    # the tiles (and so the summation grouping) follow the buckets
    assert abs(sa.norm - sb.norm) <= NORM_RTOL * sa.norm


def test_amp_large_finite_squares_are_not_an_overflow():
    """bf16 gradients of about 1e19: every square is finite in binary32
    (below 3.4e38) but the sum of two already is not.  The oracle's binary64
    sum stays finite, so the step is taken, and the GPU must agree: no
    partial sum of finite squares may overflow on its side either."""
    w = W.small((5000, 3000, 777), 2, mode="flat", align=16, dtype="bf16", op="avg")
    cfg = Z.AmpConfig(init_scale=1.0, window=0, hysteresis=1, max_norm=1.0)
    c = AmpCase(w, cfg)
    gen = torch.Generator(device="cuda").manual_seed(11)
    for t in (1, 2):
        g = []
        for q in range(2):
            mag = torch.rand(c.L, generator=gen, device="cuda") * 0.4e19 + 0.9e19
            neg = torch.rand(c.L, generator=gen, device="cuda") < 0.5
            x = torch.where(neg, -mag, mag).to(torch.bfloat16)
            x[w.phi:] = 0
            g.append(x)
        c.gpu_step(g)
        c.oracle_step_amp(g)
        torch.cuda.synchronize()
        s = c.compare_state(f"step {t}")
        assert s.overflow == 0 and s.step == t and 1e20 < s.norm < float("inf")
        c.compare(f"large squares step {t}")


def test_amp_ranks_that_own_nothing_still_decide():
    """A mask whose ranks own no element: the step still decides (norm 0, no
    overflow), counts the step and grows the scale, as the oracle does."""
    w = W.small((4000, 3000), 3, mode="round_robin", align=1, dtype="fp16", op="avg",
                rank_mask=0b100)
    c = AmpCase(w, Z.AmpConfig(init_scale=4.0, window=2, hysteresis=1))
    for t in (1, 2, 3):
        g = c.grads_scaled(t, c.ost.scale)
        c.gpu_step(g)
        c.oracle_step_amp(g)
        torch.cuda.synchronize()
        s = c.compare_state(f"call {t}")
        assert s.overflow == 0 and s.step == t and s.norm == 0.0
    assert s.scale == 8.0


@pytest.mark.parametrize("seed", range(12))
def test_amp_random_groups(seed):
    """Seeded random groups (the fused-step fuzz's draws: sizes, N up to 64,
    modes, formats, masks, buckets) under random controls: initial scales
    up to 2^24 (fp16 gradients then overflow until the scale has fallen),
    windows, tolerances and clip thresholds; five calls each.  Each draw
    also runs the bucket-reduction path (zero_reduce_scatter_bucket_amp over
    the buckets in a seeded order, then zero_step_amp_reduced), which must
    equal the fused step bit for bit."""
    from tests.test_gpu_fuzz import draw_case
    w, bucket, _, _ = draw_case(100 + seed)
    rng = np.random.default_rng(9000 + seed)
    cfg = Z.AmpConfig(init_scale=float(rng.choice([1.0, 2.0 ** 8, 2.0 ** 16, 2.0 ** 24])),
                      min_scale=1.0, window=int(rng.choice([0, 1, 2, 1000])),
                      hysteresis=int(rng.choice([1, 2, 3])),
                      max_norm=float(rng.choice([0.0, 1e-3, 0.05, 10.0])))
    c = AmpCase(w, cfg, bucket=bucket)
    red = AmpCase(w, cfg, bucket=bucket, with_oracle=False)
    B = bucket if bucket > 0 else max(1, c.plan.padded)
    order = rng.permutation(max(1, -(-c.plan.padded // B)))
    for t in range(1, 6):
        g = c.grads_scaled(t, c.ost.scale)
        c.gpu_step(g)
        c.oracle_step_amp(g)
        for b in order:
            Z.zero_reduce_scatter_bucket_amp(red.plan, g, w.op, red.gsh, HP, red.state, red.ws,
                                             int(b), rank_mask=w.mask, bucket_elems=bucket)
        Z.zero_step_amp_reduced(red.plan, red.gsh, red.master, red.m, red.v, red.full16, None,
                                HP, cfg, red.state, red.ws, rank_mask=w.mask,
                                bucket_elems=bucket, dtype=Z.ZERO_FP16 if w.dtype == "fp16"
                                else Z.ZERO_BF16)
        torch.cuda.synchronize()
        c.compare_state(f"seed {seed} call {t}")
        c.compare(f"seed {seed} call {t}")
        assert torch.equal(c.state, red.state), (seed, t)
        assert torch.equal(c.full16.view(torch.int16), red.full16.view(torch.int16)), (seed, t)
        for r in range(w.n_ranks):
            for x, y in ((c.master, red.master), (c.m, red.m), (c.v, red.v)):
                assert torch.equal(x[r].view(torch.int32), y[r].view(torch.int32)), (seed, t, r)


@pytest.mark.parametrize("seed", range(0, 12, 3))
def test_amp_random_groups_offloaded(seed):
    """The same random draws and controls through zero_offload_step_amp
    (host state, random chunk size and thread count): bit for bit the
    device-resident zero_step_amp over five calls, skipped overflows
    included."""
    from tests.test_gpu_fuzz import draw_case
    w, bucket, _, _ = draw_case(100 + seed)
    rng = np.random.default_rng(9000 + seed)
    cfg = Z.AmpConfig(init_scale=float(rng.choice([1.0, 2.0 ** 8, 2.0 ** 16, 2.0 ** 24])),
                      min_scale=1.0, window=int(rng.choice([0, 1, 2, 1000])),
                      hysteresis=int(rng.choice([1, 2, 3])),
                      max_norm=float(rng.choice([0.0, 1e-3, 0.05, 10.0])))
    ref = AmpCase(w, cfg, bucket=bucket, with_oracle=False)
    got = AmpCase(w, cfg, bucket=bucket, with_oracle=False)
    P = ref.plan.padded
    chunk = max(int(rng.integers(1, P + 2)), -(-P // 4000))
    threads = int(rng.integers(1, 9))
    S = [got.plan.shard_len(r) if (w.mask >> r) & 1 else 0 for r in range(w.n_ranks)]
    hm = [x.cpu() for x in got.master]
    hmm = [torch.zeros(n, dtype=torch.float32) for n in S]
    hv = [torch.zeros(n, dtype=torch.float32) for n in S]
    hg = [torch.zeros(n, dtype=torch.float32, pin_memory=True) if n else 0 for n in S]
    h16 = [torch.zeros(n, dtype=w.torch_dtype, pin_memory=True) if n else 0 for n in S]
    scale = cfg.init_scale
    for t in range(1, 6):
        g = ref.grads_scaled(t, scale)
        ref.gpu_step(g)
        Z.zero_offload_step_amp(got.plan, g, w.op, hg, hm, hmm, hv, h16, got.full16, HP, cfg,
                                got.state, got.ws, rank_mask=w.mask, bucket_elems=bucket,
                                chunk_elems=chunk, n_threads=threads)
        torch.cuda.synchronize()
        assert torch.equal(ref.state, got.state), (seed, t)
        assert torch.equal(ref.full16.view(torch.int16), got.full16.view(torch.int16)), (seed, t)
        for r in range(w.n_ranks):
            if S[r]:
                for x, y in ((ref.master, hm), (ref.m, hmm), (ref.v, hv)):
                    assert torch.equal(x[r].cpu().view(torch.int32), y[r].view(torch.int32)), \
                        (seed, t, r)
        scale = Z.read_amp_state(ref.state).scale

def test_amp_many_tensors_number_tiles_across_launches():
    """700 round-robin tensors: the reduction needs several launches per call
    and each numbers its tiles after the previous ones (the per-tile sums
    must land in distinct workspace slots)."""
    rng = np.random.default_rng(3)
    numel = tuple(int(x) for x in rng.integers(1, 3000, size=700))
    w = W.small(numel, 3, mode="round_robin", align=1, dtype="fp16", op="sum",
                outlier_frac=0.01)
    c = AmpCase(w, Z.AmpConfig(init_scale=256.0, window=2, hysteresis=1, max_norm=0.05))
    for t in range(1, 4):
        g = c.grads_scaled(t, c.ost.scale)
        c.gpu_step(g)
        c.oracle_step_amp(g)
        torch.cuda.synchronize()
        c.compare_state(f"many tensors call {t}")
        c.compare(f"many tensors call {t}")


def test_amp_group_without_elements_still_decides():
    """Every tensor empty: the norm is 0, the step counts, the scale grows
    after its window, exactly as the oracle's state machine says."""
    w = W.small((0, 0), 2, mode="flat", align=16, dtype="fp16", op="avg")
    c = AmpCase(w, Z.AmpConfig(init_scale=8.0, window=1, hysteresis=1))
    for t in (1, 2):
        g = [torch.empty(0, dtype=torch.float16, device="cuda") for _ in range(2)]
        c.gpu_step(g)
        c.oracle_step_amp(g)
        torch.cuda.synchronize()
        s = c.compare_state(f"empty group call {t}")
        assert s.step == t and s.norm == 0.0 and s.scale == 8.0 * 2 ** t


@pytest.mark.parametrize("bucket,mode", [(0, "flat"), (4096, "flat"), (0, "round_robin")])
def test_amp_from_reduced_shards_equals_the_fused_step(bucket, mode):
    """zero_reduce_scatter then zero_step_amp_shards == zero_step_amp, bit for
    bit, through an overflow trajectory (fp16 gradients at a scale of 2^20):
    the same decisions, state, shards and gathered parameters."""
    w = W.small((30000, 37, 4096, 3, 129), 4, mode=mode, align=16, dtype="fp16", op="avg",
                outlier_frac=0.01)
    cfg = Z.AmpConfig(init_scale=2.0 ** 20, min_scale=1.0, window=2, hysteresis=2,
                      max_norm=0.05)
    a = AmpCase(w, cfg, bucket=bucket, with_oracle=False)
    b = AmpCase(w, cfg, bucket=bucket, with_oracle=False)
    skipped = 0
    for t in range(1, 9):
        g = a.grads_scaled(t, Z.read_amp_state(a.state).scale)
        a.gpu_step(g)
        Z.zero_reduce_scatter(b.plan, g, "avg", b.gsh, bucket_elems=bucket)
        Z.zero_step_amp_shards(b.plan, b.gsh, b.master, b.m, b.v, b.full16, None, HP, cfg,
                               b.state, b.ws, bucket_elems=bucket)
        torch.cuda.synchronize()
        assert torch.equal(a.state, b.state), t
        skipped = Z.read_amp_state(a.state).skipped
        # bit patterns: overflowing steps leave NaNs in the reduced shards
        bits = lambda x: x.view(torch.int32) if x.dtype == torch.float32 else x.view(torch.int16)  # noqa: E731
        for r in range(4):
            for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v), (a.gsh, b.gsh)):
                assert torch.equal(bits(x[r]), bits(y[r])), (t, r)
        assert torch.equal(bits(a.full16), bits(b.full16)), t
    assert 0 < skipped < 8


def test_amp_shards_rejects_bad_arguments_without_launching():
    w = W.small((5000,), 2, mode="flat", align=16, dtype="bf16", op="avg")
    c = AmpCase(w, Z.AmpConfig(), with_oracle=False)
    before = Z.zero_launch_count()
    with pytest.raises(Z.ZeroError):
        Z.zero_step_amp_shards(c.plan, c.gsh, c.master, c.m, c.v, c.full16, None, HP, c.cfg,
                               c.state, c.ws[:8])
    with pytest.raises(ValueError):
        Z.zero_step_amp_shards(c.plan, c.gsh, c.master, c.m, c.v, None, None, HP, c.cfg,
                               c.state, c.ws)   # no 16-bit buffer to infer the format from
    assert Z.zero_launch_count() == before


def test_amp_workspace_too_small_is_rejected():
    w = W.small((30000,), 2, mode="flat", align=16, dtype="bf16", op="avg")
    c = AmpCase(w, Z.AmpConfig(), with_oracle=False)
    small = c.ws[:8]
    before = Z.zero_launch_count()
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_step_amp(c.plan, c.grads_scaled(1, 1.0), "avg", c.gsh, c.master, c.m, c.v,
                        c.full16, None, HP, c.cfg, c.state, small)
    assert e.value.status == Z.ZERO_ERR_INVALID and Z.zero_launch_count() == before


def test_amp_toy_model_full_size():
    """The round-robin ToyModel group (100.7M, fp16, N=4, summed, 1 % outliers)
    with DeepSpeed-like controls: scale 2^16, window 2, hysteresis 2,
    clipping at 1.0.  The oracle runs the whole group (the norm is global);
    the buffers are compared on sampled elements."""
    w = W.WORKLOADS["toy_rr"]
    cfg = Z.AmpConfig(init_scale=65536.0, min_scale=1.0, window=2, hysteresis=2, max_norm=1.0)
    c = AmpCase(w, cfg)
    F = sample_indices(w, n_random=20000)
    rank, shard = owner_of(w, F)
    applied = 0
    for t in range(1, 9):
        g = c.grads_scaled(t, c.ost.scale)
        c.gpu_step(g)
        c.oracle_step_amp(g)
        torch.cuda.synchronize()
        applied += not c.compare_state(f"call {t}").overflow
        del g
    assert applied >= 2
    for r in range(w.n_ranks):
        sel = rank == r
        it = torch.from_numpy(shard[sel]).cuda()
        assert_fp32_close(f32(c.master[r][it]), c.o_master[r][shard[sel]], f"master[{r}]")
        assert_fp32_close(f32(c.m[r][it]), c.o_m[r][shard[sel]], f"m[{r}]")
        assert_fp32_close(f32(c.v[r][it]), c.o_v[r][shard[sel]], f"v[{r}]")
    Ft = torch.from_numpy(F).cuda()
    assert_16_close(u16(c.full16[Ft]), c.o_full[F], "full16")


@pytest.mark.parametrize("numel,N,mode,A,dtype,bucket", [
    ((20000, 37, 4096, 3, 129), 4, "flat", 16, "fp16", 7000),
    ((20000, 37, 4096, 3, 129), 4, "flat", 16, "fp16", 0),
    (tuple(5 + (k * 7919) % 3001 for k in range(700)), 3, "round_robin", 1, "bf16", 300000),
    ((70001,), 8, "flat", 2, "bf16", 9000),
])
def test_bucket_reductions_then_reduced_step_equal_the_fused_step(numel, N, mode, A, dtype,
                                                                  bucket):
    """Every bucket reduced by zero_reduce_scatter_bucket_amp (last bucket
    first, as a backward pass fills them), then zero_step_amp_reduced: equal,
    bit for bit, to zero_step_amp on the replicas with the same bucket size,
    and to the oracle, through skipped overflows and clipping."""
    w = W.small(numel, N, mode=mode, align=A, dtype=dtype, op="avg", outlier_frac=0.01)
    # fp16: the first steps overflow (1 % of the entries are 100x larger)
    # until the scale has halved to 2^14; bf16 never overflows
    cfg = Z.AmpConfig(init_scale=2.0 ** 17, min_scale=1.0, window=3, hysteresis=2,
                      max_norm=0.05)
    ref = AmpCase(w, cfg, bucket=bucket)
    got = AmpCase(w, cfg, bucket=bucket, with_oracle=False)
    P = ref.plan.padded
    B = bucket if bucket > 0 else P
    nb = -(-P // B)
    for t in range(1, 9):
        g = ref.grads_scaled(t, ref.ost.scale)
        ref.gpu_step(g)
        ref.oracle_step_amp(g)
        n0 = Z.zero_launch_count()
        for b in reversed(range(nb)):
            Z.zero_reduce_scatter_bucket_amp(got.plan, g, "avg", got.gsh, HP, got.state, got.ws,
                                             b, bucket_elems=bucket)
        assert Z.zero_launch_count() - n0 >= 1
        Z.zero_step_amp_reduced(got.plan, got.gsh, got.master, got.m, got.v, got.full16, None,
                                HP, cfg, got.state, got.ws, bucket_elems=bucket)
        torch.cuda.synchronize()
        assert torch.equal(ref.state, got.state), t
        assert torch.equal(ref.full16.view(torch.int16), got.full16.view(torch.int16)), t
        for r in range(N):
            for a, b_ in ((ref.master, got.master), (ref.m, got.m), (ref.v, got.v),
                          (ref.gsh, got.gsh)):
                assert torch.equal(a[r].view(torch.int32), b_[r].view(torch.int32)), (t, r)
        ref.compare_state(f"step {t}")
        ref.compare(f"bucket reductions, step {t}")
    assert ref.ost.step >= 1
    assert ref.ost.skipped >= 1 or dtype == "bf16"


def test_bucket_amp_rejects_bad_arguments():
    w = W.small((20000, 37), 2, mode="flat", align=16, dtype="fp16", op="avg")
    cfg = Z.AmpConfig()
    c = AmpCase(w, cfg, bucket=5000, with_oracle=False)
    g = c.grads_scaled(1, 1.0)
    nb = -(-c.plan.padded // 5000)
    n0 = Z.zero_launch_count()
    for b in (-1, nb):
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_reduce_scatter_bucket_amp(c.plan, g, "avg", c.gsh, HP, c.state, c.ws, b,
                                             bucket_elems=5000)
        assert e.value.status == Z.ZERO_ERR_INVALID and "bucket" in str(e.value)
    small = torch.empty(Z.zero_amp_workspace_bytes(c.plan, bucket_elems=5000) - 16,
                        dtype=torch.uint8, device="cuda")
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_reduce_scatter_bucket_amp(c.plan, g, "avg", c.gsh, HP, c.state, small, 0,
                                         bucket_elems=5000)
    assert e.value.status == Z.ZERO_ERR_INVALID and "workspace" in str(e.value)
    assert Z.zero_launch_count() == n0


@pytest.mark.parametrize("entry", ["fused", "shards", "reduced"])
@pytest.mark.parametrize("with_full", [True, False])
def test_amp_step_writes_16bit_shards(entry, with_full):
    """The mixed-precision step with each rank's 16-bit shard as output (the
    ZeRO-3 layout), with and without the gathered flat buffer, through each
    of its three entry points: the shards, the buffer and the state equal the
    oracle's (which writes the same shard outputs), over an fp16 overflow."""
    w = W.small((20000, 37, 4096, 3, 129), 4, mode="flat", align=16, dtype="fp16", op="avg",
                outlier_frac=0.01)
    cfg = Z.AmpConfig(init_scale=2.0 ** 16, min_scale=1.0, window=2, hysteresis=1,
                      max_norm=0.05)
    bucket = 8192
    c = AmpCase(w, cfg, bucket=bucket)
    s16 = [torch.full((c.plan.shard_len(r),), 7.0, dtype=w.torch_dtype, device="cuda")
           for r in range(4)]
    o16 = [oracle.f32_to_16(np.full(c.plan.shard_len(r), 7.0, np.float32).view(np.uint32),
                            oracle.FP16) for r in range(4)]
    full = c.full16 if with_full else None
    o_full = c.o_full if with_full else None
    P = c.plan.padded
    for t in range(1, 6):
        g = c.grads_scaled(t, c.ost.scale)
        if entry == "fused":
            Z.zero_step_amp(c.plan, g, "avg", c.gsh, c.master, c.m, c.v, full, s16, HP, cfg,
                            c.state, c.ws, bucket_elems=bucket)
        elif entry == "shards":
            Z.zero_reduce_scatter(c.plan, g, "avg", c.gsh)
            Z.zero_step_amp_shards(c.plan, c.gsh, c.master, c.m, c.v, full, s16, HP, cfg,
                                   c.state, c.ws, bucket_elems=bucket)
        else:
            for b in range(-(-P // bucket)):
                Z.zero_reduce_scatter_bucket_amp(c.plan, g, "avg", c.gsh, HP, c.state, c.ws, b,
                                                 bucket_elems=bucket)
            Z.zero_step_amp_reduced(c.plan, c.gsh, c.master, c.m, c.v, full, s16, HP, cfg,
                                    c.state, c.ws, bucket_elems=bucket)
        oracle.step_amp(list(w.numel), 4, mode_code(w), w.align, dt_code(w), op_code(w),
                        [u16(x) for x in g], c.o_master, c.o_m, c.o_v, o_full, o16,
                        hp_oracle(HP), _ocfg(cfg), c.ost, w.mask)
        torch.cuda.synchronize()
        c.compare_state(f"{entry} step {t}")
        for r in range(4):
            assert_fp32_close(f32(c.master[r]), c.o_master[r], f"{entry} master[{r}] step {t}")
            assert_16_close(u16(s16[r]), o16[r], f"{entry} shard16[{r}] step {t}",
                            dtype_code=dt_code(w))
        if with_full:
            assert_16_close(u16(c.full16), c.o_full, f"{entry} full16 step {t}",
                            dtype_code=dt_code(w))
        else:
            assert not c.full16.any()               # never written
    assert c.ost.skipped >= 1 and c.ost.step >= 1


def test_reduced_path_full_size_equals_the_fused_step():
    """The BERT-base group at full size (109,482,240 elements, 8 bf16
    replicas), 5M-element buckets reduced last first, then
    zero_step_amp_reduced: every buffer and the state equal zero_step_amp's
    bit for bit over three clipped steps."""
    w = W.WORKLOADS["bert_base"]
    cfg = Z.AmpConfig(init_scale=1.0, min_scale=1.0, window=0, hysteresis=1, max_norm=0.5)
    bucket = 5_000_000
    a = AmpCase(w, cfg, bucket=bucket, with_oracle=False)
    b = AmpCase(w, cfg, bucket=bucket, with_oracle=False)
    nb = -(-a.plan.padded // bucket)
    for t in range(1, 4):
        g = a.grads_scaled(t, 1.0)
        a.gpu_step(g)
        step = Z.ReduceScatterBucketAmp(b.plan, g, "avg", b.gsh, HP, b.state, b.ws,
                                        bucket_elems=bucket)
        for k in reversed(range(nb)):
            step(k)
        Z.zero_step_amp_reduced(b.plan, b.gsh, b.master, b.m, b.v, b.full16, None, HP, cfg,
                                b.state, b.ws, bucket_elems=bucket)
        del g
        torch.cuda.synchronize()
        assert torch.equal(a.state, b.state), t
    assert Z.read_amp_state(a.state).coef < 1.0          # clipping was active
    assert torch.equal(a.full16.view(torch.int16), b.full16.view(torch.int16))
    for r in range(w.n_ranks):
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v), (a.gsh, b.gsh)):
            assert torch.equal(x[r].view(torch.int32), y[r].view(torch.int32)), r


def _host_copy(seq, pin=True):
    return [x.cpu().pin_memory() if pin else x.cpu() for x in seq]


@pytest.mark.parametrize("numel,N,mode,dtype,bucket,chunk,reduced,threads", [
    ((20000, 37, 4096, 3, 129), 4, "flat", "fp16", 7000, None, False, 0),
    ((20000, 37, 4096, 3, 129), 4, "flat", "fp16", 7000, 3001, True, 3),
    ((20000, 37, 4096, 3, 129), 4, "flat", "fp16", 0, 0, False, 2),
    ((5000, 7, 12000, 1, 333, 9000), 3, "round_robin", "bf16", 9000, 4097, True, 5),
])
def test_offload_step_amp_equals_the_device_step(numel, N, mode, dtype, bucket, chunk, reduced,
                                                 threads):
    """The mixed-precision step with the optimizer on the host: the device
    reduces (from the replicas, or bucket by bucket beforehand) and decides,
    host threads update the host state and 16-bit shards, the device gathers.
    Bit for bit like zero_step_amp on device state, and like the oracle,
    through skipped overflows (fp16) and clipping; a skipped step changes
    nothing on the host."""
    w = W.small(numel, N, mode=mode, align=16, dtype=dtype, op="avg", outlier_frac=0.01)
    cfg = Z.AmpConfig(init_scale=2.0 ** 17, min_scale=1.0, window=3, hysteresis=2,
                      max_norm=0.05)
    ref = AmpCase(w, cfg, bucket=bucket)
    got = AmpCase(w, cfg, bucket=bucket, with_oracle=False)
    S = [got.plan.shard_len(r) for r in range(N)]
    hm = _host_copy(got.master)
    hmm, hv = _host_copy(got.m, pin=False), _host_copy(got.v, pin=False)
    hg = [torch.zeros(n, dtype=torch.float32, pin_memory=True) for n in S]
    h16 = [torch.zeros(n, dtype=w.torch_dtype, pin_memory=True) for n in S]
    full = torch.zeros_like(got.full16)
    P = got.plan.padded
    B = bucket if bucket > 0 else P
    skipped_seen = False
    for t in range(1, 9):
        g = ref.grads_scaled(t, ref.ost.scale)
        ref.gpu_step(g)
        ref.oracle_step_amp(g)
        before = [x.clone() for x in hm]
        if reduced:
            for b in reversed(range(-(-P // B))):
                Z.zero_reduce_scatter_bucket_amp(got.plan, g, "avg", hg, HP, got.state, got.ws, b,
                                                 bucket_elems=bucket)
            Z.zero_offload_step_amp(got.plan, None, "avg", hg, hm, hmm, hv, h16, full, HP, cfg,
                                    got.state, got.ws, bucket_elems=bucket, chunk_elems=chunk,
                                    n_threads=threads)
        else:
            Z.zero_offload_step_amp(got.plan, g, "avg", hg, hm, hmm, hv, h16, full, HP, cfg,
                                    got.state, got.ws, bucket_elems=bucket, chunk_elems=chunk,
                                    n_threads=threads)
        torch.cuda.synchronize()
        assert torch.equal(ref.state, got.state), t
        if Z.read_amp_state(got.state).overflow:
            skipped_seen = True
            assert all(torch.equal(a, b_) for a, b_ in zip(before, hm)), t
            continue
        assert torch.equal(ref.full16.view(torch.int16), full.view(torch.int16)), t
        for r in range(N):
            for a, b_ in ((ref.master, hm), (ref.m, hmm), (ref.v, hv), (ref.gsh, hg)):
                assert torch.equal(a[r].cpu().view(torch.int32), b_[r].view(torch.int32)), (t, r)
            off = [int(x) for x in ref.o_seg[r][:, 2]]
            if mode == "flat":
                assert torch.equal(h16[r].view(torch.int16),
                                   ref.full16[off[0]:off[0] + S[r]].cpu().view(torch.int16))
        ref.compare_state(f"step {t}")
        ref.compare(f"offloaded amp step {t}")
    assert ref.ost.step >= 1
    assert skipped_seen or dtype == "bf16"


def test_offload_step_amp_rejects_bad_arguments_without_launching():
    w = W.small((20000, 37), 2, mode="flat", align=16, dtype="fp16", op="avg")
    cfg = Z.AmpConfig()
    c = AmpCase(w, cfg, with_oracle=False)
    S = [c.plan.shard_len(r) for r in range(2)]
    hm = _host_copy(c.master)
    hg = [torch.zeros(n, dtype=torch.float32, pin_memory=True) for n in S]
    h16 = [torch.zeros(n, dtype=torch.float16, pin_memory=True) for n in S]
    g = c.grads_scaled(1, 1.0)
    n0 = Z.zero_launch_count()
    with pytest.raises(Z.ZeroError, match="pinned"):
        Z.zero_offload_step_amp(c.plan, g, "avg", [x.data_ptr() for x in c.gsh], hm, hm, hm, h16,
                                c.full16, HP, cfg, c.state, c.ws)
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(Z.ZeroError, match="workspace"):
        Z.zero_offload_step_amp(c.plan, g, "avg", hg, hm, hm, hm, h16, c.full16, HP, cfg,
                                c.state, small)
    with pytest.raises(Z.ZeroError, match="chunks"):
        Z.zero_offload_step_amp(c.plan, g, "avg", hg, hm, hm, hm, h16, c.full16, HP, cfg,
                                c.state, c.ws, chunk_elems=3)
    assert Z.zero_launch_count() == n0
