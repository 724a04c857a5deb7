"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Every test here checks the oracle against something the pages or the
mathematics fix: worked numbers printed on the pages, closed forms, library
routines for special cases, brute-force invariants on tiny inputs, error
bounds.  None retypes the oracle's own formula.
"""
import itertools
import json
import math
import multiprocessing as mp
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from zero_sharded_optimizer_flatten_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# 16-bit rounding: exhaustive over every binary32 bit pattern


@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16], ids=["fp16", "bf16"])
def test_rounding_exhaustive(dtype):
    """All 2^32 binary32 inputs: the oracle's round-to-nearest-even equals
    numpy's binary16 conversion / torch's bfloat16 conversion (NaN -> NaN)."""
    oracle.build()
    from tests._cast_worker import check_range
    step = 1 << 26
    jobs = [(lo, lo + step, dtype) for lo in range(0, 1 << 32, step)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(8, os.cpu_count() or 1)) as pool:
        res = pool.map(check_range, jobs)
    assert sum(r[0] for r in res) == 0
    assert sum(r[1] for r in res) == 0


@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16], ids=["fp16", "bf16"])
def test_widening_all_16bit_values(dtype):
    """Every 16-bit pattern widens exactly as numpy / torch widen it, and every
    non-NaN value rounds back to itself."""
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.to_f32(h, dtype)
    if dtype == oracle.FP16:
        with np.errstate(invalid="ignore"):   # signalling NaNs raise the flag on some hosts
            ref = h.view(np.float16).astype(np.float32)
    else:
        ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    back = oracle.f32_to_16(got.view(np.uint32), dtype)
    assert np.array_equal(back[~nan], h[~nan])


def test_rounding_special_cases():
    """Hand-checked cases from the binary16 definition: ties to even, largest
    finite, overflow threshold, subnormal boundary."""
    def r16(x):
        return int(oracle.f32_to_16(np.array([x], np.float32).view(np.uint32), oracle.FP16)[0])
    assert r16(1.0) == 0x3C00
    assert r16(65504.0) == 0x7BFF                   # largest finite
    assert r16(65519.99) == 0x7BFF                  # below the midpoint to 2^16
    assert r16(65520.0) == 0x7C00                   # midpoint: ties to even -> overflow
    assert r16(70000.0) == 0x7C00                   # beyond the largest binade -> +inf
    assert r16(-1e30) == 0xFC00
    assert r16(2.0 ** -24) == 0x0001                # smallest subnormal
    assert r16(2.0 ** -25) == 0x0000                # tie between 0 and 2^-24 -> even (0)
    assert r16(1.5 * 2.0 ** -25) == 0x0001
    assert r16(1.0 + 2.0 ** -11) == 0x3C00           # tie -> even mantissa
    assert r16(1.0 + 3 * 2.0 ** -11) == 0x3C02       # tie -> even mantissa (up)
    assert r16(-0.0) == 0x8000


# ----------------------------------------------------------------------------
# partition plan


def _check_flat_invariants(numel, N, A):
    phi, P, S = oracle.plan_flat(numel, N, A)
    assert phi == sum(numel)
    # padding: the least multiple of N*A that holds phi
    assert P % (N * A) == 0 and phi <= P < phi + N * A
    assert S * N == P and S % A == 0
    starts = np.concatenate([[0], np.cumsum(numel)]).astype(np.int64)
    owner = -np.ones(P, np.int64)
    for r in range(N):
        seg = oracle.segments(numel, N, oracle.FLAT, A, r)
        lens = seg[:, 4] if len(seg) else np.zeros(0, np.int64)
        assert lens.sum() == S                           # equal shards
        prev_end, prev_shard = None, 0
        for k, toff, foff, soff, ln in seg:
            assert ln > 0
            if k >= 0:
                assert 0 <= toff and toff + ln <= numel[k]
                assert foff == starts[k] + toff          # flat index from the tensor walk
            else:
                assert foff >= phi                        # padding lies past phi
            assert soff == prev_shard                     # shard is the segments in order
            if prev_end is not None:
                assert foff == prev_end                   # one contiguous flat range
            prev_end, prev_shard = foff + ln, soff + ln
            assert (owner[foff:foff + ln] == -1).all()    # disjoint
            owner[foff:foff + ln] = r
    assert (owner >= 0).all()                             # covering
    assert (np.diff(owner) >= 0).all()                    # rank r's range before rank r+1's


def test_flat_plan_brute_force_tiny():
    """Every tensor-size list of length <= 3 with sizes 0..5, N in 1..8,
    A in {1, 2, 8, 16}: equal, aligned, contiguous, rank-ordered, disjoint
    and covering shards with the least padding."""
    for n in range(0, 4):
        for numel in itertools.product(range(0, 6), repeat=n):
            for N in range(1, 9):
                for A in (1, 2, 8, 16):
                    _check_flat_invariants(list(numel), N, A)


def test_flat_plan_configs():
    """The five parameter groups: sizes from the published shapes."""
    expect = {"tiny_mlp": (1053706, 1053760, 263440), "bert_base": (109482240, 109482240,
              13685280), "llama7b_rank0": (6738415616, 6738415616, 842301952),
              "llama13b_layer": (212336640, 212336640, 26542080),
              "llama13b_full_layer": (317204480, 317204480, 39650560)}
    for key, (phi, P, S) in expect.items():
        w = W.WORKLOADS[key]
        assert oracle.plan_flat(list(w.numel), w.n_ranks, w.align) == (phi, P, S)
    _check_flat_invariants(list(W.WORKLOADS["tiny_mlp"].numel), 4, 16)


def test_round_robin_example_from_page():
    """Page example: 4 GPUs, params 0,4,8 -> GPU 0 ... 3,7,11 -> GPU 3."""
    g = json.load(open(os.path.join(GOLDEN, "rr_example.json")))
    N = g["world_size"]
    numel = [3] * 12
    for r in range(N):
        seg = oracle.segments(numel, N, oracle.ROUND_ROBIN, 1, r)
        owned = sorted(int(k) for k in seg[:, 0])
        assert owned == sorted(int(i) for i, o in g["owners"].items() if o == r)


def test_round_robin_brute_force_tiny():
    for n in range(0, 6):
        for numel in itertools.product([0, 1, 3], repeat=n):
            for N in range(1, 6):
                starts = np.concatenate([[0], np.cumsum(numel)]).astype(np.int64)
                covered = np.zeros(int(sum(numel)), np.int64)
                for r in range(N):
                    seg = oracle.segments(list(numel), N, oracle.ROUND_ROBIN, 1, r)
                    shard = 0
                    for k, toff, foff, soff, ln in seg:
                        assert k % N == r and toff == 0 and ln == numel[k]
                        assert foff == starts[k] and soff == shard
                        shard += ln
                        covered[foff:foff + ln] += 1
                assert (covered == 1).all()


def test_round_robin_toy_model_shards():
    """Inter-tensor imbalance of the 12-layer ToyModel at N=4 ("ZeRO 优化器",
    ZeRO-3 的分片方式: whole tensors per owner, so shards are uneven)."""
    w = W.WORKLOADS["toy_rr"]
    lens = [oracle.shard_len(list(w.numel), 4, oracle.ROUND_ROBIN, 1, r) for r in range(4)]
    assert lens == [12 * 4096 * 1024 + 1024 * 10, 12 * 4096 + 10, 12 * 1024 * 4096, 12 * 1024]
    assert sum(lens) == w.phi == 100734986


# ----------------------------------------------------------------------------
# memory model


def test_memory_model_closed_forms():
    """The per-rank totals exactly as the pages print them (16Φ, 4Φ + 12Φ/N,
    2Φ + 14Φ/N, 16Φ/N), as exact rationals over a grid of Φ and N that
    includes N not dividing Φ; the table's rows must add up to its totals."""
    g = json.load(open(os.path.join(GOLDEN, "memory_closed_forms.json")))
    phis = [0, 1, 7, 1000, 4096 * 3 + 5, 109482240, 6738415616, 10 ** 12 + 39]
    ranks = [1, 2, 3, 4, 5, 7, 8, 13, 64]
    assert [c["stage"] for c in g["stages"]] == [0, 1, 2, 3]
    for c in g["stages"]:
        for k in ("whole", "split"):
            assert c["params"][k] + c["grads"][k] + c["optimizer"][k] == c["total"][k]
        assert c["total"]["whole"] + c["total"]["split"] == 16     # one rank holds 16 B/param
        for phi in phis:
            for N in ranks:
                want = c["total"]["whole"] * phi + Fraction(c["total"]["split"] * phi, N)
                assert Fraction(*oracle.memory_bytes(c["stage"], phi, N)) == want, \
                    (c["name"], phi, N)


def test_memory_model_closed_forms_by_hand():
    """The same forms at a few hand-worked points (Φ = 1000, N = 8):
    16000, 4000 + 1500, 2000 + 1750, 2000 bytes; and Φ = 10, N = 3, where
    N does not divide Φ: 160, 40 + 40, 20 + 140/3, 160/3."""
    mb = lambda s, phi, N: Fraction(*oracle.memory_bytes(s, phi, N))  # noqa: E731
    assert [mb(s, 1000, 8) for s in range(4)] == [16000, 5500, 3750, 2000]
    assert [mb(s, 10, 3) for s in range(4)] == [160, 80, Fraction(200, 3), Fraction(160, 3)]


def test_memory_model_worked_numbers():
    g = json.load(open(os.path.join(GOLDEN, "memory_worked_numbers.json")))
    mb = lambda s, phi, N: Fraction(*oracle.memory_bytes(s, phi, N))
    for c in g["cases"]:
        phi, N = c["phi"], c["n_ranks"]
        if c["kind"] == "stage0_total":
            assert mb(0, phi, N) == (c["params_bytes"] + c["grads_bytes"] + c["moments_bytes"]
                                     + c["master_bytes_per_param"] * phi)
        elif c["kind"] == "stage2_minus_stage3":
            assert mb(2, phi, N) - mb(3, phi, N) == (c["params_full_bytes"]
                                                    - c["params_sharded_bytes"])
        elif c["kind"] == "stage1_optimizer_saving":
            # optimizer-state bytes of an unsharded rank, read off the stage-1
            # saving at N=2 (half of it is saved there)
            opt_full = 2 * (mb(0, phi, 2) - mb(1, phi, 2))
            saving = (mb(0, phi, N) - mb(1, phi, N)) / opt_full
            assert saving == Fraction(c["saving"]).limit_denominator(1000)
        elif c["kind"] == "stage0_optimizer_share":
            assert mb(0, phi, N) == c["total_per_param"] * phi
            opt_full = 2 * (mb(0, phi, 2) - mb(1, phi, 2))
            assert opt_full / mb(0, phi, N) == Fraction(c["optimizer_share"]).limit_denominator(100)
        else:
            raise AssertionError(c["kind"])


# ----------------------------------------------------------------------------
# reduction


def _as16(x, dtype):
    t = torch.tensor(x, dtype=torch.float64).to(torch.float32)
    t = t.to(torch.float16 if dtype == oracle.FP16 else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8])
def test_reduce_exact_on_small_integers(dtype, N):
    """Small integers times 2^-10 sum exactly in binary32: the sum equals the
    exact rational sum; the average is the correctly rounded quotient."""
    rng = np.random.default_rng(N)
    k = rng.integers(-64, 65, size=(N, 257))
    g16 = _as16(k * 2.0 ** -10, dtype)
    exact = k.sum(axis=0) * 2.0 ** -10                 # exact in binary64
    s = oracle.reduce_elements(g16, dtype, oracle.SUM)
    assert np.array_equal(s.astype(np.float64), exact)
    a = oracle.reduce_elements(g16, dtype, oracle.AVG)
    # binary32 division of binary32 operands == binary64 quotient rounded once
    # more (53 >= 2*24+2 bits, so the double rounding is innocuous)
    assert np.array_equal(a, (exact / N).astype(np.float32))


def test_reduce_follows_rank_order():
    """Replicas 1, 2^-24, 2^-24 (exact in binary16): in rank order 0, 1, 2 the
    binary32 sum stays 1 (each 1 + 2^-24 is a tie that rounds to even); any
    order that adds the two small terms first gives 1 + 2^-23.  The average is
    that sum divided by 3 once (not the sum of thirds)."""
    g = np.stack([_as16([1.0], oracle.FP16), _as16([2.0 ** -24], oracle.FP16),
                  _as16([2.0 ** -24], oracle.FP16)])
    s = oracle.reduce_elements(g, oracle.FP16, oracle.SUM)
    assert s[0] == np.float32(1.0)
    assert np.float32(1.0) + (np.float32(2.0 ** -24) + np.float32(2.0 ** -24)) != s[0]
    a = oracle.reduce_elements(g, oracle.FP16, oracle.AVG)
    assert a[0] == np.float32(1.0) / np.float32(3.0)
    thirds = (np.float32(1.0) / np.float32(3.0) + np.float32(2.0 ** -24) / np.float32(3.0)) \
        + np.float32(2.0 ** -24) / np.float32(3.0)
    assert thirds != a[0]
    # the reverse rank order reaches the other value
    r = oracle.reduce_elements(g[::-1].copy(), oracle.FP16, oracle.SUM)
    assert r[0] == np.float32(1.0 + 2.0 ** -23)


@pytest.mark.parametrize("N", [2, 4, 8, 16])
def test_reduce_error_bound(N):
    """Random fp16 gradients: |binary32 recursive sum - exact| <= gamma_{N-1} sum|g|."""
    rng = np.random.default_rng(100 + N)
    x = rng.normal(0, 1e-2, size=(N, 4096))
    x[rng.random(x.shape) < 0.01] *= 100
    g16 = _as16(x, oracle.FP16)
    vals = g16.view(np.float16).astype(np.float64)
    exact = np.array([math.fsum(vals[:, i]) for i in range(vals.shape[1])])
    u = 2.0 ** -24
    gamma = (N - 1) * u / (1 - (N - 1) * u)
    got = oracle.reduce_elements(g16, oracle.FP16, oracle.SUM).astype(np.float64)
    assert (np.abs(got - exact) <= gamma * np.abs(vals).sum(axis=0) + 1e-300).all()
    # and it is not the exact sum everywhere (the reduction really rounds)
    got_avg = oracle.reduce_elements(g16, oracle.FP16, oracle.AVG).astype(np.float64)
    assert (np.abs(got_avg - exact / N) <= (gamma + 2 * u) * np.abs(vals).sum(axis=0) / N
            + 1e-300).all()


# ----------------------------------------------------------------------------
# AdamW


def _torch_adamw(p0, grads, hp):
    p = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([p], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=hp.weight_decay, foreach=False, fused=False)
    for g in grads:
        p.grad = torch.from_numpy(g.copy())
        opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


def _normwise(a, b):
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    return np.max(np.abs(a - b)) / np.max(np.abs(b))


@pytest.mark.parametrize("gscale", [1e-2, 1e-8], ids=["g1e-2", "g~eps"])
@pytest.mark.parametrize("hp", [oracle.hparams(), oracle.hparams(lr=1e-4, weight_decay=0.0),
                                oracle.hparams(lr=3e-2, beta1=0.8, beta2=0.95, eps=1e-6,
                                               weight_decay=0.1)],
                         ids=["cfg", "wd0", "aggressive"])
def test_adamw_matches_torch(hp, gscale):
    """N=1, ten steps: master/m/v agree with torch.optim.AdamW (fp32 CPU,
    single-tensor path) to 1e-6 of their magnitude.  torch orders a few
    operations differently (a lerp for m, addcdiv for the update), so single
    elements that cancel to near zero differ by a few ulps of the operands;
    the comparison is therefore norm-wise.  Gradients of the size of eps make
    the placement of eps decide the update."""
    rng = np.random.default_rng(5)
    n = 20000
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    grads = [rng.normal(0, gscale, n).astype(np.float32) for _ in range(10)]
    master, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t, g in enumerate(grads, start=1):
        oracle.adamw_elements(g, master, m, v, oracle.BF16, hp, t)
    tp, tm, tv = _torch_adamw(p0, grads, hp)
    assert _normwise(master, tp) <= 1e-6
    assert _normwise(m, tm) <= 1e-6
    assert _normwise(v, tv) <= 1e-6


def test_adamw_constant_gradient_closed_form():
    """With a constant gradient g, the bias-corrected moments are g and g^2 at
    every step, so p_t = p_{t-1} (1 - lr wd) - lr g / (|g| + eps)."""
    hp = oracle.hparams()
    rng = np.random.default_rng(9)
    n = 4096
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-2, n).astype(np.float32)
    master, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    ref = p0.astype(np.float64)
    for t in range(1, 6):
        oracle.adamw_elements(g, master, m, v, oracle.FP16, hp, t)
        gd = g.astype(np.float64)
        ref = ref * (1 - hp.lr * hp.weight_decay) - hp.lr * gd / (np.abs(gd) + hp.eps)
        # a few binary32 roundings per step on |update| ~ lr
        assert np.max(np.abs(master - ref)) <= 8 * t * 2.0 ** -24 * (hp.lr + np.abs(ref).max())


def test_adamw_first_step_decays_before_the_update():
    """First step (m = v = 0, t = 1) at a large learning rate and decay:
    p1 = p0 (1 - lr wd) - lr g / (|g| + eps).  Decaying after the update
    instead would give (p0 - lr g / (|g| + eps)) (1 - lr wd), which differs
    here by lr^2 wd = 5e-3 per unit gradient sign."""
    hp = oracle.hparams(lr=0.1, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.5)
    rng = np.random.default_rng(13)
    n = 4096
    p0 = rng.normal(0, 1.0, n).astype(np.float32)
    g = rng.normal(0, 1e-2, n).astype(np.float32)
    master, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle.adamw_elements(g, master, m, v, oracle.FP16, hp, 1)
    pd, gd = p0.astype(np.float64), g.astype(np.float64)
    u = hp.lr * gd / (np.abs(gd) + hp.eps)
    first = pd * (1 - hp.lr * hp.weight_decay) - u
    after = (pd - u) * (1 - hp.lr * hp.weight_decay)
    err = np.abs(master - first)
    assert err.max() <= 16 * 2.0 ** -24 * (np.abs(first).max() + hp.lr)
    assert np.abs(after - first).min() >= 1e-3 > err.max()


def test_adamw_zero_gradient_decays_only():
    hp = oracle.hparams()
    rng = np.random.default_rng(11)
    p0 = rng.normal(0, 0.02, 1000).astype(np.float32)
    master, m, v = p0.copy(), np.zeros(1000, np.float32), np.zeros(1000, np.float32)
    for t in range(1, 8):
        oracle.adamw_elements(np.zeros(1000, np.float32), master, m, v, oracle.FP16, hp, t)
    assert not m.any() and not v.any()
    # the decay factor is one binary32 number; seven products round once each
    d32 = float(np.float32(1 - hp.lr * hp.weight_decay))
    ref = p0.astype(np.float64) * d32 ** 7
    assert np.max(np.abs(master - ref) / np.abs(ref)) <= 7.01 * 2.0 ** -24


def test_cast_of_update_is_rounding_of_master():
    """The 16-bit output is the master rounded to nearest even (torch's cast)."""
    hp = oracle.hparams()
    rng = np.random.default_rng(12)
    n = 5000
    g16 = _as16(rng.normal(0, 1e-2, (4, n)), oracle.BF16)
    master = rng.normal(0, 0.02, n).astype(np.float32)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    out = np.zeros(n, np.uint16)
    oracle.update_elements(g16, master, m, v, oracle.BF16, oracle.AVG, hp, 1, out16=out)
    ref = torch.from_numpy(master).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, ref)


# ----------------------------------------------------------------------------
# the whole step: partition invariance


def _run_sharded(w, steps, hp):
    """Oracle step over the plan with N virtual ranks."""
    mode = oracle.FLAT if w.mode == "flat" else oracle.ROUND_ROBIN
    L = oracle.flat_len(list(w.numel), w.n_ranks, mode, w.align)
    dt = oracle.FP16 if w.dtype == "fp16" else oracle.BF16
    op = oracle.AVG if w.op == "avg" else oracle.SUM
    p16 = W.params16(w, "cpu", L).view(torch.int16).numpy().view(np.uint16)
    shards = []
    for r in range(w.n_ranks):
        seg = oracle.segments(list(w.numel), w.n_ranks, mode, w.align, r)
        S = int(seg[:, 4].sum()) if len(seg) else 0
        mst = np.zeros(S, np.float32)
        for k, toff, foff, soff, ln in seg:
            mst[soff:soff + ln] = oracle.to_f32(p16[foff:foff + ln], dt)
        shards.append((mst, np.zeros(S, np.float32), np.zeros(S, np.float32), seg))
    full = np.zeros(L, np.uint16)
    for t in range(1, steps + 1):
        grads = [W.grads16(w, t, q, "cpu", 0, L).view(torch.int16).numpy().view(np.uint16)
                 for q in range(w.n_ranks)]
        oracle.step(list(w.numel), w.n_ranks, mode, w.align, dt, op, grads,
                    [s[0] for s in shards], [s[1] for s in shards], [s[2] for s in shards],
                    full, None, hp, t)
    return p16, shards, full


def _run_unsharded(w, steps, hp):
    """The same group as ONE flat buffer: reduce all N replicas, plain AdamW."""
    dt = oracle.FP16 if w.dtype == "fp16" else oracle.BF16
    op = oracle.AVG if w.op == "avg" else oracle.SUM
    mode = oracle.FLAT if w.mode == "flat" else oracle.ROUND_ROBIN
    L = oracle.flat_len(list(w.numel), w.n_ranks, mode, w.align)
    p16 = W.params16(w, "cpu", L).view(torch.int16).numpy().view(np.uint16)
    master = oracle.to_f32(p16, dt)
    m, v = np.zeros_like(master), np.zeros_like(master)
    out = np.zeros(p16.size, np.uint16)
    for t in range(1, steps + 1):
        grads = np.stack([W.grads16(w, t, q, "cpu", 0, L).view(torch.int16).numpy()
                          .view(np.uint16) for q in range(w.n_ranks)])
        g = oracle.reduce_elements(grads, dt, op)
        oracle.adamw_elements(g, master, m, v, dt, hp, t, out16=out)
    return master, m, v, out


@pytest.mark.parametrize("numel,N,mode,A,dtype,op", [
    ((1000, 37, 4096, 3, 129), 4, "flat", 16, "fp16", "avg"),
    ((1000, 37, 4096, 3, 129), 3, "flat", 2, "bf16", "sum"),
    ((1000, 37, 4096, 3, 129), 8, "flat", 8, "bf16", "avg"),
    ((1000, 37, 4096, 3, 129), 5, "round_robin", 1, "fp16", "sum"),
    ((7,), 8, "flat", 16, "fp16", "avg"),
])
def test_partition_invariance(numel, N, mode, A, dtype, op):
    """Sharded over N virtual ranks == plain AdamW on the whole flat buffer,
    bit for bit ([ZeRO-2 blog] §4.3: each rank updates its partition with no
    other rank's optimizer state)."""
    hp = oracle.hparams()
    w = W.small(numel, N, mode=mode, align=A, dtype=dtype, op=op, outlier_frac=0.01)
    p16, shards, full = _run_sharded(w, 3, hp)
    master, m, v, out = _run_unsharded(w, 3, hp)
    for mst, mm, vv, seg in shards:
        for k, toff, foff, soff, ln in seg:
            assert np.array_equal(mst[soff:soff + ln].view(np.uint32),
                                  master[foff:foff + ln].view(np.uint32))
            assert np.array_equal(mm[soff:soff + ln], m[foff:foff + ln])
            assert np.array_equal(vv[soff:soff + ln], v[foff:foff + ln])
    assert np.array_equal(full, out)
    if mode == "flat":
        phi = sum(numel)
        assert not full[phi:].any()                      # padding gathers as +0


def test_unfused_composition_equals_step():
    """reduce_scatter -> AdamW on each shard -> allgather == step."""
    hp = oracle.hparams()
    w = W.small((300, 5000, 17), 4, mode="round_robin", align=1, dtype="fp16", op="sum")
    p16, shards, full = _run_sharded(w, 1, hp)
    # recompute step 1 through the unfused pieces
    dt, mode = oracle.FP16, oracle.ROUND_ROBIN
    grads = [W.grads16(w, 1, q, "cpu", 0, full.size).view(torch.int16).numpy().view(np.uint16)
             for q in range(4)]
    outs, sh16 = [], []
    for r in range(4):
        seg = oracle.segments(list(w.numel), 4, mode, 1, r)
        S = int(seg[:, 4].sum()) if len(seg) else 0
        outs.append(np.zeros(S, np.float32))
    oracle.reduce_scatter(list(w.numel), 4, mode, 1, dt, oracle.SUM, grads, outs)
    full2 = np.zeros_like(full)
    for r in range(4):
        seg = oracle.segments(list(w.numel), 4, mode, 1, r)
        mst = np.zeros(outs[r].size, np.float32)
        for k, toff, foff, soff, ln in seg:
            mst[soff:soff + ln] = oracle.to_f32(p16[foff:foff + ln], dt)
        m, v = np.zeros_like(mst), np.zeros_like(mst)
        o16 = np.zeros(mst.size, np.uint16)
        oracle.adamw_elements(outs[r], mst, m, v, dt, hp, 1, out16=o16)
        sh16.append(o16)
        assert np.array_equal(mst, shards[r][0])
    oracle.allgather(list(w.numel), 4, mode, 1, sh16, full2)
    assert np.array_equal(full, full2)
