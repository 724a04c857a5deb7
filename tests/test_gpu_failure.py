"""Failure detection without a GPU fault: a kernel's bounded wait that runs
out raises the device error word, zero_sync reports ZERO_ERR_TIMEOUT once,
and the context stays usable for the next step."""
import gc

import pytest
import torch

from tests._harness import Case, hp_oracle
from zero_sharded_optimizer_flatten_gb300 import workloads as W
from zero_sharded_optimizer_flatten_gb300 import zero as Z

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda_cleanup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    gc.collect()
    torch.cuda.synchronize()


def test_bounded_wait_reports_timeout_and_context_survives():
    Z.zero_sync()                                  # nothing pending
    Z.zero_selftest_wait_timeout(20_000_000)      # 20 ms on a barrier nothing completes
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_sync()
    assert e.value.status == Z.ZERO_ERR_TIMEOUT
    Z.zero_sync()                                  # reported once, then cleared
    # the context is intact: a normal step still matches the oracle
    w = W.small((5000, 33), 4, mode="flat", align=16, dtype="bf16", op="avg")
    c = Case(w)
    g = c.grads(1)
    Z.zero_step(c.plan, g, "avg", c.master, c.m, c.v, c.full16, None, Z.AdamW(), 1)
    c.oracle_step(g, 1, hp_oracle(Z.AdamW()))
    Z.zero_sync()
    c.compare("after timeout")


def test_timeout_on_a_side_stream():
    s = torch.cuda.Stream()
    Z.zero_selftest_wait_timeout(5_000_000, stream=s)
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_sync(s)
    assert e.value.status == Z.ZERO_ERR_TIMEOUT
