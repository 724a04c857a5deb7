"""Shared set-up for the GPU parity tests: buffers on the device for the CUDA
path, host arrays for the oracle, both fed from the seeded workloads."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from zero_sharded_optimizer_flatten_gb300 import workloads as W
from zero_sharded_optimizer_flatten_gb300 import zero as Z

# Pass criteria: fp32 state within 1e-6 relative (element-wise, denominators
# floored at the smallest normal), 16-bit parameters within 1 ulp.
FP32_RTOL = 1e-6
ULP16 = 1


def flat_len(w: W.Workload) -> int:
    """Length of the gathered flat buffer (tail padding included), from the
    oracle's plan."""
    return oracle.flat_len(list(w.numel), w.n_ranks, mode_code(w), w.align)


def dt_code(w: W.Workload) -> int:
    return oracle.FP16 if w.dtype == "fp16" else oracle.BF16


def op_code(w: W.Workload) -> int:
    return oracle.AVG if w.op == "avg" else oracle.SUM


def mode_code(w: W.Workload) -> int:
    return oracle.FLAT if w.mode == "flat" else oracle.ROUND_ROBIN


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def assert_fp32_close(got: np.ndarray, ref: np.ndarray, what: str, rtol: float = FP32_RTOL):
    got = np.asarray(got, np.float32)
    ref = np.asarray(ref, np.float32)
    assert got.shape == ref.shape, what
    nan_ok = np.isnan(got) == np.isnan(ref)
    assert nan_ok.all(), f"{what}: NaN mismatch"
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    fin = np.isfinite(r)
    assert np.array_equal(g[~fin & ~np.isnan(r)], r[~fin & ~np.isnan(r)]), f"{what}: inf mismatch"
    err = np.abs(g[fin] - r[fin]) / np.maximum(np.abs(r[fin]), 2.0 ** -126)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= rtol, f"{what}: max relative error {worst:.3g} > {rtol}"


def key16(x: np.ndarray) -> np.ndarray:
    """Monotone integer key of 16-bit float bit patterns (adjacent values
    differ by 1; +0 and -0 share key 0)."""
    x = x.astype(np.int64)
    return np.where(x & 0x8000, -(x & 0x7FFF), x)


def is_nan16(x: np.ndarray, dtype_code: int) -> np.ndarray:
    """NaN bit patterns of binary16 (dtype_code 0: exponent field 0x1f) or
    bfloat16 (dtype_code 1: exponent field 0xff), non-zero mantissa."""
    x = x.astype(np.int64)
    if dtype_code == 0:
        return ((x & 0x7C00) == 0x7C00) & ((x & 0x03FF) != 0)
    return ((x & 0x7F80) == 0x7F80) & ((x & 0x007F) != 0)


def assert_16_close(got: np.ndarray, ref: np.ndarray, what: str, ulps: int = ULP16,
                    dtype_code: int = None):
    """Within `ulps` ulp; a NaN must meet a NaN (any payload: the pages fix no
    NaN encoding, and the hardware's conversion picks its own)."""
    assert got.shape == ref.shape, what
    if dtype_code is not None:
        ng, nr = is_nan16(got, dtype_code), is_nan16(ref, dtype_code)
        assert np.array_equal(ng, nr), f"{what}: NaN positions differ"
        got, ref = got[~ng], ref[~nr]
    d = np.abs(key16(got) - key16(ref))
    worst = int(d.max()) if d.size else 0
    assert worst <= ulps, f"{what}: {worst} ulp apart (> {ulps})"


class Case:
    """Device buffers of one workload plus the oracle's host copy of them."""

    def __init__(self, w: W.Workload, device="cuda", with_oracle=True, layer: int = 0):
        self.w, self.dev = w, device
        self.plan = Z.zero_plan_partitions(list(w.numel), w.n_ranks, w.mode, w.align)
        self.L = flat_len(w)
        assert self.plan.padded == self.L
        self.p16 = W.params16(w, device, self.L, layer=layer)
        self.full16 = torch.zeros(self.L, dtype=w.torch_dtype, device=device)
        mask = w.mask
        self.master, self.m, self.v = [], [], []
        for r in range(w.n_ranks):
            n = self.plan.shard_len(r) if (mask >> r) & 1 else 0
            self.master.append(torch.empty(n, dtype=torch.float32, device=device))
            self.m.append(torch.empty(n, dtype=torch.float32, device=device))
            self.v.append(torch.empty(n, dtype=torch.float32, device=device))
        Z.zero_init_shards(self.plan, self.p16, self.master, self.m, self.v, rank_mask=mask)
        self.o = None
        if with_oracle:
            self._oracle_init()

    def _oracle_init(self):
        w = self.w
        p16 = u16(self.p16)
        self.o_master, self.o_m, self.o_v, self.o_seg = [], [], [], []
        for r in range(w.n_ranks):
            seg = oracle.segments(list(w.numel), w.n_ranks, mode_code(w), w.align, r)
            S = int(seg[:, 4].sum()) if len(seg) else 0
            mst = np.zeros(S, np.float32)
            for k, toff, foff, soff, ln in seg:
                mst[soff:soff + ln] = oracle.to_f32(p16[foff:foff + ln], dt_code(w))
            self.o_master.append(mst)
            self.o_m.append(np.zeros(S, np.float32))
            self.o_v.append(np.zeros(S, np.float32))
            self.o_seg.append(seg)
        self.o_full = np.zeros(self.L, np.uint16)
        self.o = True

    def grads(self, t: int):
        return [W.grads16(self.w, t, q, self.dev, 0, self.L) for q in range(self.w.n_ranks)]

    def oracle_step(self, grads, t: int, hp: oracle.Hparams, mask=None):
        w = self.w
        g = [u16(x) for x in grads]
        mask = w.mask if mask is None else mask
        oracle.step(list(w.numel), w.n_ranks, mode_code(w), w.align, dt_code(w), op_code(w), g,
                    self.o_master, self.o_m, self.o_v, self.o_full, None, hp, t, mask)

    def compare(self, what: str, mask=None):
        w = self.w
        mask = w.mask if mask is None else mask
        for r in range(w.n_ranks):
            if not (mask >> r) & 1:
                continue
            assert_fp32_close(f32(self.master[r]), self.o_master[r], f"{what} master[{r}]")
            assert_fp32_close(f32(self.m[r]), self.o_m[r], f"{what} m[{r}]")
            assert_fp32_close(f32(self.v[r]), self.o_v[r], f"{what} v[{r}]")
        assert_16_close(u16(self.full16), self.o_full, f"{what} full16",
                        dtype_code=dt_code(self.w))


def hp_oracle(h: Z.AdamW) -> oracle.Hparams:
    return oracle.hparams(h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)


def owner_of(w: W.Workload, flat_idx: np.ndarray):
    """(rank, shard index) of each flat index, from the oracle's segments."""
    rank = -np.ones(flat_idx.size, np.int64)
    shard = -np.ones(flat_idx.size, np.int64)
    for r in range(w.n_ranks):
        seg = oracle.segments(list(w.numel), w.n_ranks, mode_code(w), w.align, r)
        for k, toff, foff, soff, ln in seg:
            hit = (flat_idx >= foff) & (flat_idx < foff + ln)
            rank[hit] = r
            shard[hit] = soff + flat_idx[hit] - foff
    return rank, shard


def sample_indices(w: W.Workload, n_random: int = 20000, seed: int = 99, extra=()):
    """Seeded random flat indices plus every boundary the kernels care about:
    shard and tensor starts/ends, the tail padding, 2048-element tile edges
    next to shard starts, and caller-given extras (bucket edges)."""
    L = flat_len(w)
    rng = np.random.default_rng(seed)
    # random points inside the flat ranges of the masked ranks only
    ranges = []
    for r in range(w.n_ranks):
        if (w.mask >> r) & 1:
            seg = oracle.segments(list(w.numel), w.n_ranks, mode_code(w), w.align, r)
            ranges += [(int(f), int(f + n)) for _, _, f, _, n in seg]
    lens = np.array([b - a for a, b in ranges], np.int64)
    pick = rng.choice(len(ranges), size=n_random, p=lens / lens.sum())
    offs = (rng.random(n_random) * lens[pick]).astype(np.int64)
    pts = [np.array([ranges[i][0] for i in pick], np.int64) + offs]
    edges = [0, L - 1]
    starts = np.concatenate([[0], np.cumsum(np.asarray(w.numel, np.int64))])
    edges += list(starts)
    for r in range(w.n_ranks):
        seg = oracle.segments(list(w.numel), w.n_ranks, mode_code(w), w.align, r)
        for k, toff, foff, soff, ln in seg:
            edges += [foff, foff + ln - 1, foff + 2048, foff + 2047]
    edges += list(extra)
    e = np.asarray(edges, np.int64)
    e = np.concatenate([e - 1, e, e + 1])
    idx = np.unique(np.concatenate(pts + [e]))
    return idx[(idx >= 0) & (idx < L)]
