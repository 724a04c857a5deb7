"""Pins of the oracle's mixed-precision step (loss scaling, overflow skip,
global-norm clipping) to facts outside itself: the plain step it must reduce
to, exact power-of-two scaling, torch's clip_grad_norm_ + AdamW, and the
loss-scale trajectory the configuration keys describe."""
import math

import numpy as np
import pytest
import torch

import oracle
from zero_sharded_optimizer_flatten_gb300 import workloads as W

NUMEL = (1000, 37, 4096, 3, 129)


def _flat_len(w):
    mode = oracle.FLAT if w.mode == "flat" else oracle.ROUND_ROBIN
    return oracle.flat_len(list(w.numel), w.n_ranks, mode, w.align)


def _setup(w):
    mode = oracle.FLAT if w.mode == "flat" else oracle.ROUND_ROBIN
    dt = oracle.FP16 if w.dtype == "fp16" else oracle.BF16
    p16 = W.params16(w, "cpu", _flat_len(w)).view(torch.int16).numpy().view(np.uint16)
    master, m, v = [], [], []
    for r in range(w.n_ranks):
        seg = oracle.segments(list(w.numel), w.n_ranks, mode, w.align, r)
        S = int(seg[:, 4].sum()) if len(seg) else 0
        mst = np.zeros(S, np.float32)
        for k, toff, foff, soff, ln in seg:
            mst[soff:soff + ln] = oracle.to_f32(p16[foff:foff + ln], dt)
        master.append(mst)
        m.append(np.zeros(S, np.float32))
        v.append(np.zeros(S, np.float32))
    return mode, dt, master, m, v, np.zeros(_flat_len(w), np.uint16)


def _grads(w, t, scale=1.0):
    """Replicas drawn in binary32, multiplied by `scale`, rounded to 16 bits."""
    out = []
    for q in range(w.n_ranks):
        x = W.grads16(w, t, q, "cpu", 0, _flat_len(w)).float() * scale
        out.append(x.to(w.torch_dtype).view(torch.int16).numpy().view(np.uint16))
    return out


def _op(w):
    return oracle.AVG if w.op == "avg" else oracle.SUM


@pytest.mark.parametrize("mode,N", [("flat", 4), ("round_robin", 3)])
def test_unit_scale_without_clipping_is_the_plain_step(mode, N):
    w = W.small(NUMEL, N, mode=mode, align=16, dtype="bf16", op="avg")
    hp = oracle.hparams()
    mode_c, dt, ma, ma_m, ma_v, full_a = _setup(w)
    _, _, mb, mb_m, mb_v, full_b = _setup(w)
    cfg = oracle.amp_config(init_scale=1.0, window=0, hysteresis=1, max_norm=0.0)
    st = oracle.amp_init(cfg)
    for t in (1, 2, 3):
        g = _grads(w, t)
        oracle.step(list(w.numel), N, mode_c, 16, dt, oracle.AVG, g, ma, ma_m, ma_v, full_a, None,
                    hp, t)
        oracle.step_amp(list(w.numel), N, mode_c, 16, dt, oracle.AVG, g, mb, mb_m, mb_v, full_b,
                        None, hp, cfg, st)
    assert st.step == 3 and st.overflow == 0 and st.coef == 1.0
    for r in range(N):
        assert np.array_equal(ma[r].view(np.uint32), mb[r].view(np.uint32))
        assert np.array_equal(ma_v[r], mb_v[r])
    assert np.array_equal(full_a, full_b)


def test_power_of_two_scale_unscales_exactly():
    """fp16 gradients that are exact multiples 2^10 x (the unscaled ones):
    the scaled step equals the unscaled step bit for bit."""
    w = W.small(NUMEL, 4, mode="flat", align=16, dtype="fp16", op="sum", grad_sigma=1e-3)
    hp = oracle.hparams()
    mode_c, dt, ma, ma_m, ma_v, full_a = _setup(w)
    _, _, mb, mb_m, mb_v, full_b = _setup(w)
    S = 1024.0
    cfg = oracle.amp_config(init_scale=S, window=0, hysteresis=1, max_norm=0.0)
    st = oracle.amp_init(cfg)
    for t in (1, 2):
        g = _grads(w, t)
        gs = []
        for x in g:   # exact scaling of binary16 values by 2^10 (no overflow at sigma 1e-3)
            y = x.view(np.float16).astype(np.float32) * np.float32(S)
            assert np.isfinite(y).all()
            gs.append(y.astype(np.float16).view(np.uint16))
            assert np.array_equal(gs[-1].view(np.float16).astype(np.float32) / np.float32(S),
                                  x.view(np.float16).astype(np.float32))
        oracle.step(list(w.numel), 4, mode_c, 16, dt, oracle.SUM, g, ma, ma_m, ma_v, full_a, None,
                    hp, t)
        oracle.step_amp(list(w.numel), 4, mode_c, 16, dt, oracle.SUM, gs, mb, mb_m, mb_v, full_b,
                        None, hp, cfg, st)
    assert st.coef == np.float32(1 / S)
    for r in range(4):
        assert np.array_equal(ma[r].view(np.uint32), mb[r].view(np.uint32))
    assert np.array_equal(full_a, full_b)


@pytest.mark.parametrize("max_norm", [0.05, 1e-3])
def test_clipping_matches_torch(max_norm):
    """N=1: oracle(step_amp) == torch clip_grad_norm_ then torch.optim.AdamW,
    both run in binary64 on the same gradients, within 1e-6 of the magnitude."""
    w = W.small((20000,), 1, mode="flat", align=16, dtype="bf16", op="sum", grad_sigma=1e-2)
    hp = oracle.hparams()
    mode_c, dt, mst, m, v, full = _setup(w)
    cfg = oracle.amp_config(init_scale=1.0, window=0, hysteresis=1, max_norm=max_norm)
    st = oracle.amp_init(cfg)
    p = torch.nn.Parameter(torch.from_numpy(mst[0].copy()).double())
    opt = torch.optim.AdamW([p], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=hp.weight_decay, foreach=False)
    clipped = 0
    for t in (1, 2, 3):
        g = _grads(w, t)
        gf = torch.from_numpy(oracle.to_f32(g[0][:20000], dt)).double()
        p.grad = gf.clone()
        norm = torch.nn.utils.clip_grad_norm_([p], max_norm)
        clipped += float(norm) > max_norm
        opt.step()
        oracle.step_amp(list(w.numel), 1, mode_c, 16, dt, oracle.SUM, g, mst, m, v, full, None, hp,
                        cfg, st)
        # squares rounded to binary32 (relative error <= 2^-24 each)
        assert abs(st.norm - float(norm)) <= 2.0 ** -24 * float(norm)
    assert clipped == 3
    ref = p.detach().numpy()
    assert np.max(np.abs(mst[0][:20000] - ref)) <= 1e-6 * np.max(np.abs(ref))
    tm = opt.state[p]["exp_avg"].numpy()
    assert np.max(np.abs(m[0][:20000] - tm)) <= 1e-6 * np.max(np.abs(tm))


def test_overflow_skips_and_halves_after_hysteresis():
    w = W.small(NUMEL, 4, mode="flat", align=16, dtype="fp16", op="avg")
    hp = oracle.hparams()
    mode_c, dt, mst, m, v, full = _setup(w)
    cfg = oracle.amp_config(init_scale=4096.0, min_scale=1024.0, window=1000, hysteresis=2)
    st = oracle.amp_init(cfg)
    g = _grads(w, 1)
    oracle.step_amp(list(w.numel), 4, mode_c, 16, dt, oracle.AVG, g, mst, m, v, full, None, hp,
                    cfg, st)
    assert st.step == 1 and st.overflow == 0
    before = [x.copy() for x in mst], [x.copy() for x in v], full.copy()
    bad = _grads(w, 2)
    bad[2][123] = 0x7C00        # +inf in rank 2's replica
    expect_scale = [4096.0, 2048.0, 1024.0, 1024.0]   # tolerance 2: first overflow keeps S
    for k in range(4):
        oracle.step_amp(list(w.numel), 4, mode_c, 16, dt, oracle.AVG, bad, mst, m, v, full, None,
                        hp, cfg, st)
        assert st.overflow == 1 and st.step == 1 and st.skipped == k + 1
        assert st.scale == expect_scale[k]
        assert not np.isfinite(st.norm)
    for r in range(4):
        assert np.array_equal(mst[r], before[0][r]) and np.array_equal(v[r], before[1][r])
    assert np.array_equal(full, before[2])
    bad[2][123] = 0x7E00        # NaN is caught the same way
    oracle.step_amp(list(w.numel), 4, mode_c, 16, dt, oracle.AVG, bad, mst, m, v, full, None, hp,
                    cfg, st)
    assert st.overflow == 1 and st.skipped == 5


def test_scale_grows_every_window_of_good_steps():
    w = W.small((4096,), 2, mode="flat", align=16, dtype="fp16", op="avg", grad_sigma=1e-4)
    hp = oracle.hparams()
    mode_c, dt, mst, m, v, full = _setup(w)
    cfg = oracle.amp_config(init_scale=8.0, window=3, hysteresis=2)
    st = oracle.amp_init(cfg)
    scales = []
    for t in range(1, 8):
        oracle.step_amp([4096], 2, mode_c, 16, dt, oracle.AVG, _grads(w, t), mst, m, v, full,
                        None, hp, cfg, st)
        scales.append(st.scale)
    # closed form: S after k good steps = S0 * 2^floor(k / window)
    assert scales == [8.0 * 2 ** (k // 3) for k in range(1, 8)]
    assert st.step == 7 and st.good_steps == 1 and st.hysteresis_left == 2


# ----------------------------------------------------------------------------
# the squared norm: binary32 squares of the reduced gradient, summed in binary64
#
# Reading (the pages give only the fp16 / gradient_clipping configuration
# keys, "ZeRO ... 实操" (wmrh.cn) §3.1, §3.3): the reduced gradient and
# every operation on it are binary32 (fp16 training with fp32 gradients and
# master weights), so each square g*g is the binary32 product -- the same
# product the second-moment update forms; the squares are added in binary64
# so that the norm does not depend on the partition or the order.  Each pin
# below fails under the other plausible readings: exact (binary64) squares,
# or a binary32 sum.


def _norm_case(values_by_rank, dtype, op=oracle.SUM, max_norm=0.0):
    """One step of the oracle's mixed-precision step on a single tensor whose
    replicas hold the given 16-bit values (binary64 numbers, exact in the
    format); returns the state after it."""
    N = len(values_by_rank)
    n = len(values_by_rank[0])
    td = torch.float16 if dtype == oracle.FP16 else torch.bfloat16
    g = []
    for vals in values_by_rank:
        t = torch.tensor(vals, dtype=torch.float64)
        h = t.to(td)
        assert torch.equal(h.double(), t), "value not exact in the 16-bit format"
        g.append(h.view(torch.int16).numpy().view(np.uint16).copy())
    L = oracle.flat_len([n], N, oracle.FLAT, 16)
    g = [np.concatenate([x, np.zeros(L - n, np.uint16)]) for x in g]
    master, m, v = [], [], []
    for r in range(N):
        S = oracle.shard_len([n], N, oracle.FLAT, 16, r)
        master.append(np.zeros(S, np.float32))
        m.append(np.zeros(S, np.float32))
        v.append(np.zeros(S, np.float32))
    cfg = oracle.amp_config(init_scale=1.0, window=0, hysteresis=1, max_norm=max_norm)
    st = oracle.amp_init(cfg)
    oracle.step_amp([n], N, oracle.FLAT, 16, dtype, op, g, master, m, v,
                    np.zeros(L, np.uint16), None, oracle.hparams(), cfg, st)
    return st


def test_norm_squares_are_binary32_products():
    """Replicas 1 and 2^-12 sum to g = 1 + 2^-12 (exact in binary32); its
    exact square 1 + 2^-11 + 2^-24 is a tie in binary32 and rounds to the
    even 1 + 2^-11.  Over 4096 elements the squared norm is 4096 + 2 exactly;
    exact squares would give 4096 + 2 + 2^-12."""
    n = 4096
    st = _norm_case([[1.0] * n, [2.0 ** -12] * n], oracle.FP16)
    assert st.overflow == 0 and st.step == 1
    assert st.norm == math.sqrt(n + 2)
    assert st.norm != math.sqrt(n + 2 + 2.0 ** -12)
    assert abs(math.sqrt(n + 2 + 2.0 ** -12) - math.sqrt(n + 2)) > 1e-9 * st.norm


def test_norm_sum_is_binary64():
    """One element 2^12 (square 2^24) then 1000 elements 1: a binary32 running
    sum stays at 2^24 (each +1 is a tie that rounds back to even), the
    binary64 sum is 2^24 + 1000 exactly."""
    st = _norm_case([[4096.0] + [1.0] * 1000], oracle.FP16)
    assert st.overflow == 0
    assert st.norm == math.sqrt(2.0 ** 24 + 1000)


def test_overflow_is_a_binary32_square_out_of_range():
    """bf16 gradients: 2^63 squares to 2^126 (finite); 2^64 squares to 2^128,
    beyond binary32, so the step is skipped as an overflow (its exact square
    would be a finite binary64 number)."""
    st = _norm_case([[2.0 ** 63] + [0.0] * 15], oracle.BF16)
    assert st.overflow == 0 and st.norm == 2.0 ** 63
    st = _norm_case([[2.0 ** 64] + [0.0] * 15], oracle.BF16)
    assert st.overflow == 1 and st.step == 0 and st.skipped == 1


def test_large_finite_squares_sum_beyond_binary32():
    """Four bf16 gradients 1.5 x 2^63: each binary32 square 2.25 x 2^126 is
    finite, their sum 9 x 2^126 is beyond binary32 but not binary64, so the
    step is not an overflow and the norm is 3 x 2^63 exactly."""
    st = _norm_case([[1.5 * 2.0 ** 63] * 4 + [0.0] * 12], oracle.BF16)
    assert st.overflow == 0 and st.step == 1
    assert st.norm == 3 * 2.0 ** 63
