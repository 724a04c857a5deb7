"""ZeRO-Offload's CPU optimizer (zero_cpu_adamw_shard_step) against the
oracle, on the host (no GPU): host threads must give the oracle's AdamW and
16-bit rounding bit for bit, for any thread count."""
import numpy as np
import pytest

import oracle
from zero_sharded_optimizer_flatten_gb300 import _build
from zero_sharded_optimizer_flatten_gb300 import zero as Z


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()


@pytest.mark.parametrize("dtype", [Z.ZERO_BF16, Z.ZERO_FP16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("mode,N,threads", [("flat", 4, 0), ("flat", 3, 1), ("round_robin", 4, 5)])
def test_cpu_adamw_matches_oracle(dtype, mode, N, threads):
    numel = [30011, 37, 4096, 3, 129, 70000]
    plan = Z.zero_plan_partitions(numel, N, mode, 16)
    rng = np.random.default_rng(N * 10 + threads)
    S = [plan.shard_len(r) for r in range(N)]
    hp = Z.AdamW(lr=2e-3, weight_decay=0.05)
    ohp = oracle.hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay)
    mst = [rng.normal(0, 0.02, n).astype(np.float32) for n in S]
    m = [np.zeros(n, np.float32) for n in S]
    v = [np.zeros(n, np.float32) for n in S]
    om, omm, ov = [x.copy() for x in mst], [x.copy() for x in m], [x.copy() for x in v]
    out = [np.zeros(n, np.uint16) for n in S]
    for t in (1, 2, 3):
        g = [rng.normal(0, 1e-2, n).astype(np.float32) for n in S]
        g[0][:5] = [0.0, -0.0, 1e-30, -1e-38, 3e4]        # zero, subnormal-range, large
        Z.zero_cpu_adamw_shard_step(plan, mst, m, v, g, out, hp, t, dtype, n_threads=threads)
        for r in range(N):
            o16 = np.zeros(S[r], np.uint16)
            oracle.adamw_elements(g[r], om[r], omm[r], ov[r], dtype, ohp, t, out16=o16)
            assert np.array_equal(mst[r].view(np.uint32), om[r].view(np.uint32)), (t, r)
            assert np.array_equal(m[r].view(np.uint32), omm[r].view(np.uint32))
            assert np.array_equal(v[r].view(np.uint32), ov[r].view(np.uint32))
            assert np.array_equal(out[r], o16)


def test_cpu_adamw_rejects_bad_arguments():
    plan = Z.zero_plan_partitions([1000], 2, "flat", 16)
    x = [np.zeros(plan.shard_len(r), np.float32) for r in range(2)]
    with pytest.raises(Z.ZeroError):
        Z.zero_cpu_adamw_shard_step(plan, x, x, x, x, None, Z.AdamW(), 0, Z.ZERO_BF16)
    with pytest.raises(Z.ZeroError):
        Z.zero_cpu_adamw_shard_step(plan, x, x, x, [x[0], 0], None, Z.AdamW(), 1, Z.ZERO_BF16)



def _nan_mask(u, bits, dtype=None):
    """NaN positions of binary32 (bits 32) or 16-bit patterns of `dtype`."""
    if bits == 32:
        return np.isnan(u.view(np.float32))
    exp_mask, man_mask = (0x7F80, 0x007F) if dtype == Z.ZERO_BF16 else (0x7C00, 0x03FF)
    return ((u & exp_mask) == exp_mask) & ((u & man_mask) != 0)


def _same_or_both_nan(got, want, bits, dtype=None):
    """Bit-equal, except that a NaN need only be a NaN on both sides (its
    payload follows the host's NaN propagation, which IEEE leaves open)."""
    ng, nw = _nan_mask(got, bits, dtype), _nan_mask(want, bits, dtype)
    assert np.array_equal(ng, nw)
    assert np.array_equal(got[~ng], want[~nw])


@pytest.mark.parametrize("dtype", [Z.ZERO_BF16, Z.ZERO_FP16], ids=["bf16", "fp16"])
def test_cpu_adamw_non_finite_values_and_no_cast(dtype):
    """Infinite and NaN gradients, gradients whose square overflows binary32,
    master values past the fp16 range and a bf16 rounding tie: the host loop
    (vectorised, with the cast in the same pass) gives the oracle's IEEE
    results; without a 16-bit output it updates the state identically."""
    plan = Z.zero_plan_partitions([4099], 1, "flat", 1)
    n = plan.shard_len(0)
    rng = np.random.default_rng(7)
    hp = Z.AdamW(lr=1e-3, weight_decay=0.01)
    ohp = oracle.hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay)
    mst = rng.normal(0, 0.02, n).astype(np.float32)
    mst[:6] = [7e4, -7e4, 65519.0, 65520.0, 1.0 + 2.0 ** -8, 3e38]
    g = rng.normal(0, 1e-2, n).astype(np.float32)
    g[6:12] = [np.inf, -np.inf, np.nan, 3e38, -2e19, 0.0]
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    om, omm, ov = mst.copy(), m.copy(), v.copy()
    nm, nmm, nv = mst.copy(), m.copy(), v.copy()
    out = np.zeros(n, np.uint16)
    o16 = np.zeros(n, np.uint16)
    for t in (1, 2):
        Z.zero_cpu_adamw_shard_step(plan, [mst], [m], [v], [g], [out], hp, t, dtype)
        Z.zero_cpu_adamw_shard_step(plan, [nm], [nmm], [nv], [g], None, hp, t, dtype)
        oracle.adamw_elements(g, om, omm, ov, dtype, ohp, t, out16=o16)
        for got, want in ((mst, om), (m, omm), (v, ov), (nm, om), (nmm, omm), (nv, ov)):
            _same_or_both_nan(got.view(np.uint32), want.view(np.uint32), 32)
        _same_or_both_nan(out, o16, 16, dtype)
    assert np.isnan(mst[6:9]).all()          # inf / inf and NaN reach the master
    assert np.isinf(v[9:11]).all()           # the squares of 3e38 and 2e19 overflow
    assert np.isfinite(mst[9:11]).all()      # ... so the step m / den is 0
