"""Seeded random parameter groups through the fused step, compared with the
oracle over whole buffers.

Each case draws a tensor-size mix (empty tensors, a few elements, sizes that
straddle the 2048-element tiles, up to 150k), the number of virtual ranks
(1 to 64, the compile-time paths 1..8 and the generic one), the partition
mode and alignment, the 16-bit format, sum or average, a random rank mask,
a bucket size, whether the ZeRO-3 shard outputs are written, and one of a
few AdamW settings.  Two steps each; the bar is the usual one (fp32 state
within 1e-6 relative, 16-bit parameters within 1 ulp) plus the shard
outputs bit-identical to the oracle's.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
from tests._harness import (Case, assert_16_close, assert_fp32_close, dt_code, f32, hp_oracle,
                            mode_code, op_code, u16)
from zero_sharded_optimizer_flatten_gb300 import workloads as W
from zero_sharded_optimizer_flatten_gb300 import zero as Z

pytestmark = pytest.mark.gpu

N_CASES = 40
HPS = [Z.AdamW(), Z.AdamW(lr=3e-2, beta1=0.8, beta2=0.95, eps=1e-6, weight_decay=0.1),
       Z.AdamW(lr=1e-4, weight_decay=0.0)]


@pytest.fixture(autouse=True)
def _cuda_cleanup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def draw_case(seed: int):
    rng = np.random.default_rng(5000 + seed)
    n = int(rng.integers(1, 13))
    numel = []
    for kind in rng.choice(5, size=n, p=[0.08, 0.2, 0.3, 0.35, 0.07]):
        lo, hi = [(0, 1), (1, 8), (8, 301), (301, 20001), (20001, 150001)][kind]
        numel.append(int(rng.integers(lo, hi)))
    if sum(numel) == 0:
        numel[0] = 1
    N = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 12, 16, 33, 64],
                       p=[.06, .12, .1, .12, .08, .08, .14, .06, .06, .08, .05, .05]))
    mode = "flat" if rng.random() < 0.7 else "round_robin"
    align = int(rng.choice([1, 2, 4, 8, 16, 32, 128])) if mode == "flat" else 1
    dtype = "fp16" if rng.random() < 0.5 else "bf16"
    op = "avg" if rng.random() < 0.6 else "sum"
    bits = rng.random(N) < 0.7
    if not bits.any():
        bits[int(rng.integers(N))] = True
    mask = sum(1 << r for r in range(N) if bits[r])
    phi = sum(numel)
    # at most about 40 buckets (each bucket is at least one launch)
    bucket = 0 if rng.random() < 0.6 else int(rng.integers(max(1, phi // 40), 2 * phi + 2))
    shard_out = bool(rng.random() < 0.4)
    hp = HPS[int(rng.integers(len(HPS)))]
    w = W.small(tuple(numel), N, mode=mode, align=align, dtype=dtype, op=op,
                outlier_frac=0.01, seed=seed, rank_mask=mask if mask != (1 << N) - 1 else None)
    return w, bucket, shard_out, hp


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_group_matches_oracle(seed):
    w, bucket, shard_out, hp = draw_case(seed)
    what = (f"seed {seed}: numel {w.numel} N={w.n_ranks} {w.mode} A={w.align} {w.dtype} "
            f"{w.op} mask={w.mask:#x} bucket={bucket} shards={shard_out}")
    c = Case(w)
    S = [c.plan.shard_len(r) if (w.mask >> r) & 1 else 0 for r in range(w.n_ranks)]
    s16 = [torch.full((n,), 0x7777, dtype=torch.int16, device="cuda").view(w.torch_dtype)
           for n in S] if shard_out else None
    o16 = [np.zeros(n, np.uint16) for n in S] if shard_out else None
    for t in (1, 2):
        g = c.grads(t)
        Z.zero_step(c.plan, g, w.op, c.master, c.m, c.v, c.full16, s16, hp, t,
                    rank_mask=w.mask, bucket_elems=bucket)
        oracle.step(list(w.numel), w.n_ranks, mode_code(w), w.align, dt_code(w), op_code(w),
                    [u16(x) for x in g], c.o_master, c.o_m, c.o_v, c.o_full, o16,
                    hp_oracle(hp), t, w.mask)
    torch.cuda.synchronize()
    c.compare(what)
    if shard_out:
        for r in range(w.n_ranks):
            if S[r]:
                assert_16_close(u16(s16[r]), o16[r], f"{what} shard16[{r}]",
                                dtype_code=dt_code(w))
    # the plan the library built is the oracle's, bit for bit
    for r in range(w.n_ranks):
        seg = oracle.segments(list(w.numel), w.n_ranks, mode_code(w), w.align, r)
        assert np.array_equal(c.plan.segments(r), seg), what


def test_fuzz_covers_the_dispatch_paths():
    """The drawn cases reach every kind of launch the step has."""
    draws = [draw_case(s) for s in range(N_CASES)]
    Ns = {w.n_ranks for w, *_ in draws}
    assert Ns & {1, 2, 3, 4, 5, 7, 8} and Ns & {9, 12, 16, 33, 64}
    assert {w.mode for w, *_ in draws} == {"flat", "round_robin"}
    assert {w.dtype for w, *_ in draws} == {"fp16", "bf16"}
    assert {w.op for w, *_ in draws} == {"sum", "avg"}
    assert any(b for _, b, _, _ in draws) and any(not b for _, b, _, _ in draws)
    assert any(s for _, _, s, _ in draws)
    assert any(w.rank_mask is not None for w, *_ in draws)
    assert any(0 in w.numel for w, *_ in draws)


@pytest.mark.parametrize("seed", range(0, N_CASES, 2))
def test_random_group_unfused_calls_match_oracle(seed):
    """The unfused calls on the same random draws (masks, buckets, N up to
    64 so the generic kernels too): zero_reduce_scatter bit for bit against
    the oracle's reduce-scatter; zero_adamw_shard_step (16-bit shard output
    on or off) and zero_allgather of those shards against the oracle's step;
    two steps."""
    w, bucket, shard_out, hp = draw_case(seed)
    what = (f"seed {seed}: numel {w.numel} N={w.n_ranks} {w.mode} A={w.align} {w.dtype} "
            f"{w.op} mask={w.mask:#x} bucket={bucket} shards={shard_out}")
    c = Case(w)
    S = [c.plan.shard_len(r) if (w.mask >> r) & 1 else 0 for r in range(w.n_ranks)]
    gsh = [torch.empty(n, dtype=torch.float32, device="cuda") for n in S]
    s16 = [torch.empty(n, dtype=w.torch_dtype, device="cuda") for n in S]
    for t in (1, 2):
        g = c.grads(t)
        Z.zero_reduce_scatter(c.plan, g, w.op, gsh, rank_mask=w.mask, bucket_elems=bucket)
        torch.cuda.synchronize()
        orc = [np.zeros(n, np.float32) for n in S]
        oracle.reduce_scatter(list(w.numel), w.n_ranks, mode_code(w), w.align, dt_code(w),
                              op_code(w), [u16(x) for x in g], orc, w.mask)
        for r in range(w.n_ranks):
            if S[r]:
                assert np.array_equal(f32(gsh[r]).view(np.uint32), orc[r].view(np.uint32)), \
                    f"{what} grad shard {r} step {t}"
        Z.zero_adamw_shard_step(c.plan, c.master, c.m, c.v, gsh, s16 if shard_out else None, hp,
                                t, rank_mask=w.mask,
                                dtype=Z.ZERO_FP16 if w.dtype == "fp16" else Z.ZERO_BF16)
        if shard_out:
            Z.zero_allgather(c.plan, s16, c.full16, rank_mask=w.mask)
        oracle.step(list(w.numel), w.n_ranks, mode_code(w), w.align, dt_code(w), op_code(w),
                    [u16(x) for x in g], c.o_master, c.o_m, c.o_v, c.o_full, None,
                    hp_oracle(hp), t, w.mask)
    torch.cuda.synchronize()
    for r in range(w.n_ranks):
        if (w.mask >> r) & 1:
            assert_fp32_close(f32(c.master[r]), c.o_master[r], f"{what} master[{r}]")
            assert_fp32_close(f32(c.m[r]), c.o_m[r], f"{what} m[{r}]")
            assert_fp32_close(f32(c.v[r]), c.o_v[r], f"{what} v[{r}]")
    if shard_out:
        assert_16_close(u16(c.full16), c.o_full, f"{what} full16", dtype_code=dt_code(w))


@pytest.mark.parametrize("seed", range(1, N_CASES, 4))
def test_random_group_offload_step(seed):
    """zero_offload_step on the same random draws (masks, N up to 64, both
    layouts), with a random chunk size and thread count: the host state,
    the host 16-bit shards and the gathered buffer against the oracle's
    step, two steps."""
    w, _, _, hp = draw_case(seed)
    rng = np.random.default_rng(9000 + seed)
    c = Case(w)
    P = c.plan.padded
    # 0: one chunk; else a chunk size that leaves at most 4000 chunks
    chunk = max(int(rng.integers(1, P + 2)), -(-P // 4000)) if rng.random() < 0.8 else 0
    threads = int(rng.integers(1, 9))
    what = (f"seed {seed}: numel {w.numel} N={w.n_ranks} {w.mode} A={w.align} {w.dtype} "
            f"{w.op} mask={w.mask:#x} chunk={chunk} threads={threads}")
    S = [c.plan.shard_len(r) if (w.mask >> r) & 1 else 0 for r in range(w.n_ranks)]
    hm = [x.cpu() for x in c.master]
    hmm = [torch.zeros(n, dtype=torch.float32) for n in S]
    hv = [torch.zeros(n, dtype=torch.float32) for n in S]
    hg = [torch.zeros(n, dtype=torch.float32, pin_memory=True) if n else 0 for n in S]
    h16 = [torch.zeros(n, dtype=w.torch_dtype, pin_memory=True) if n else 0 for n in S]
    for t in (1, 2):
        g = c.grads(t)
        Z.zero_offload_step(c.plan, g, w.op, hg, hm, hmm, hv, h16, c.full16, hp, t,
                            rank_mask=w.mask, chunk_elems=chunk, n_threads=threads)
        oracle.step(list(w.numel), w.n_ranks, mode_code(w), w.align, dt_code(w), op_code(w),
                    [u16(x) for x in g], c.o_master, c.o_m, c.o_v, c.o_full, None,
                    hp_oracle(hp), t, w.mask)
    torch.cuda.synchronize()
    for r in range(w.n_ranks):
        if not S[r]:
            continue
        assert_fp32_close(hm[r].numpy(), c.o_master[r], f"{what} master[{r}]")
        assert_fp32_close(hmm[r].numpy(), c.o_m[r], f"{what} m[{r}]")
        assert_fp32_close(hv[r].numpy(), c.o_v[r], f"{what} v[{r}]")
        seg = c.o_seg[r]
        want = np.concatenate([c.o_full[f:f + n] for _, _, f, _, n in seg])
        assert_16_close(u16(h16[r]), want, f"{what} shard16[{r}]", dtype_code=dt_code(w))
    assert_16_close(u16(c.full16), c.o_full, f"{what} full16", dtype_code=dt_code(w))
