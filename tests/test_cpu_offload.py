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
