"""zero_floor_probe, the measurement floor of the fused step: it must launch
the step's shape (one launch per bucket) and leave every buffer's value as it
was, except the 16-bit output, which receives the master rounded to 16 bits
(what a step leaves there anyway); arguments are checked like zero_step's."""
import gc

import pytest
import torch

import oracle
from tests._harness import Case, assert_16_close, dt_code, u16
from zero_sharded_optimizer_flatten_gb300 import workloads as W
from zero_sharded_optimizer_flatten_gb300 import zero as Z

pytestmark = pytest.mark.gpu

HP = Z.AdamW()


@pytest.fixture(autouse=True)
def _cuda_cleanup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("numel,N,mode,dtype,bucket", [
    ((30000, 37, 4096, 3, 129), 4, "flat", "bf16", 0),
    ((30000, 37, 4096, 3, 129), 3, "round_robin", "fp16", 0),
    ((50000, 7, 9000), 8, "flat", "fp16", 12000),
])
def test_floor_probe_changes_no_value(numel, N, mode, dtype, bucket):
    w = W.small(numel, N, mode=mode, align=16, dtype=dtype, op="avg")
    c = Case(w)
    g = c.grads(1)
    Z.zero_step(c.plan, g, "avg", c.master, c.m, c.v, c.full16, None, HP, 1, bucket_elems=bucket)
    torch.cuda.synchronize()
    before = [[x.clone() for x in c.master], [x.clone() for x in c.m], [x.clone() for x in c.v]]
    full_before = c.full16.clone()
    c.full16.zero_()
    for kind in (0, 1):
        n0 = Z.zero_launch_count()
        Z.zero_floor_probe(c.plan, kind, g, c.master, c.m, c.v, c.full16, bucket_elems=bucket)
        assert Z.zero_launch_count() > n0
    torch.cuda.synchronize()
    assert not c.full16.any()                       # kinds 0 and 1 store nothing
    Z.zero_floor_probe(c.plan, 2, g, c.master, c.m, c.v, c.full16, bucket_elems=bucket)
    torch.cuda.synchronize()
    for now, then in zip([c.master, c.m, c.v], before):
        for r in range(N):
            assert torch.equal(now[r], then[r])
    assert torch.equal(c.full16, full_before)
    # the stored 16-bit output is the oracle's rounding of the master
    c.oracle_step(g, 1, oracle.hparams())
    assert_16_close(u16(c.full16), c.o_full, "full16", dtype_code=dt_code(w))


def test_floor_probe_rejects_bad_arguments():
    w = W.small((4096,), 2, mode="flat", align=16, dtype="bf16", op="avg")
    c = Case(w, with_oracle=False)
    g = c.grads(1)
    n0 = Z.zero_launch_count()
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_floor_probe(c.plan, 3, g, c.master, c.m, c.v, c.full16)
    assert e.value.status == Z.ZERO_ERR_INVALID
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_floor_probe(c.plan, 1, g, c.master, c.m, c.v, c.full16.data_ptr() + 2)
    assert e.value.status == Z.ZERO_ERR_ALIGN
    assert Z.zero_launch_count() == n0
