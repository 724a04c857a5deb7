"""Host-side tests of the C-ABI library (no GPU needed).

The library must load, export every call include/zero.h declares, build the
same partition plan as the oracle bit for bit, and reject bad arguments with
the documented status before it touches the device.
"""
import ctypes
import itertools
import os
import re

import numpy as np
import pytest

import oracle
from zero_sharded_optimizer_flatten_gb300 import _build
from zero_sharded_optimizer_flatten_gb300 import workloads as W
from zero_sharded_optimizer_flatten_gb300 import zero as Z

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return Z.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "zero.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[\w\s\*]*?\b(zero_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert "zero_step" in names and "zero_plan_partitions" in names and len(names) >= 15
    for n in names:
        assert hasattr(L, n), f"libzero.so does not export {n}"


def test_version_and_counter(L):
    assert "sm_103a" in Z.zero_version()
    assert Z.zero_launch_count() >= 0


def _oracle_mode(mode):
    return oracle.FLAT if mode == "flat" else oracle.ROUND_ROBIN


def _compare_plan(numel, N, mode, A):
    plan = Z.zero_plan_partitions(numel, N, mode, A)
    om = _oracle_mode(mode)
    if mode == "flat":
        phi, P, S = oracle.plan_flat(numel, N, A)
        assert (plan.phi, plan.padded) == (phi, P)
    else:
        assert (plan.phi, plan.padded) == (sum(numel), sum(numel))
    for r in range(N):
        lib_seg = plan.segments(r)
        orc_seg = oracle.segments(numel, N, om, A, r)
        assert np.array_equal(lib_seg, orc_seg), (numel, N, mode, A, r)
        assert plan.shard_len(r) == (int(orc_seg[:, 4].sum()) if len(orc_seg) else 0)


def test_plan_matches_oracle_tiny(L):
    for n in range(1, 4):
        for numel in itertools.product([0, 1, 5, 17], repeat=n):
            for N in (1, 2, 3, 4, 8):
                for A in (1, 2, 16):
                    _compare_plan(list(numel), N, "flat", A)
                _compare_plan(list(numel), N, "round_robin", 1)


@pytest.mark.parametrize("key", list(W.WORKLOADS))
def test_plan_matches_oracle_configs(L, key):
    w = W.WORKLOADS[key]
    _compare_plan(list(w.numel), w.n_ranks, w.mode, w.align)
    # the other partition mode on the same group, too
    _compare_plan(list(w.numel), w.n_ranks, "round_robin" if w.mode == "flat" else "flat", 16)


def test_memory_bytes_matches_oracle(L):
    for stage in range(4):
        for phi in (0, 1, 7, 110_000_000, 6_738_415_616):
            for N in (1, 2, 3, 8, 64):
                assert Z.zero_memory_bytes(stage, phi, N) == oracle.memory_bytes(stage, phi, N)
    with pytest.raises(Z.ZeroError):
        Z.zero_memory_bytes(4, 10, 2)


# ----------------------------------------------------------------------------
# argument checking: every failure is reported before anything is launched

def test_plan_rejects_bad_arguments(L):
    bad = [([], 2, "flat", 16), ([4], 0, "flat", 16), ([4], 65, "flat", 16),
           ([4], 2, "flat", 3), ([4], 2, "flat", 8192), ([-1, 4], 2, "flat", 16),
           ([4], 2, 7, 16)]
    for numel, N, mode, A in bad:
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_plan_partitions(numel, N, mode, A)
        assert e.value.status == Z.ZERO_ERR_INVALID
    out = ctypes.c_void_p()
    assert L.zero_plan_partitions(None, 1, 1, 0, 16, ctypes.byref(out)) == Z.ZERO_ERR_INVALID
    assert L.zero_plan_partitions((ctypes.c_int64 * 1)(4), 1, 1, 0, 16, None) == Z.ZERO_ERR_INVALID


def _arr(vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def test_step_rejects_bad_arguments_without_launching(L):
    plan = Z.zero_plan_partitions([100, 28], 2, "flat", 16)
    good = 1 << 20  # a 16-byte-aligned non-NULL address; nothing is ever launched here
    g = _arr([good, good])
    st = _arr([good, good])
    hp = Z.AdamW().c()
    before = Z.zero_launch_count()

    def step(**kw):
        a = dict(plan=plan.handle, grads=g, dtype=Z.ZERO_BF16, op=Z.ZERO_REDUCE_AVG, master=st,
                 m=st, v=st, full=good, o16=None, hp=ctypes.byref(hp), step=1, mask=3,
                 bucket=0, stream=None)
        a.update(kw)
        return L.zero_step(a["plan"], a["grads"], a["dtype"], a["op"], a["master"], a["m"],
                           a["v"], a["full"], a["o16"], a["hp"], a["step"], a["mask"],
                           a["bucket"], a["stream"])

    assert step(plan=None) == Z.ZERO_ERR_INVALID
    assert step(mask=0) == Z.ZERO_ERR_INVALID
    assert step(mask=4) == Z.ZERO_ERR_INVALID            # rank 2 of a 2-rank plan
    assert step(dtype=5) == Z.ZERO_ERR_INVALID
    assert step(op=9) == Z.ZERO_ERR_INVALID
    assert step(step=0) == Z.ZERO_ERR_INVALID
    assert step(hp=None) == Z.ZERO_ERR_INVALID
    assert step(grads=None) == Z.ZERO_ERR_INVALID
    assert step(grads=_arr([good, 0])) == Z.ZERO_ERR_INVALID   # every replica is needed
    assert step(master=_arr([good, 0])) == Z.ZERO_ERR_INVALID
    assert step(grads=_arr([good, good + 2])) == Z.ZERO_ERR_ALIGN
    assert step(v=_arr([good + 8, good])) == Z.ZERO_ERR_ALIGN
    assert step(full=good + 4) == Z.ZERO_ERR_ALIGN
    assert step(o16=_arr([good + 2, 0])) == Z.ZERO_ERR_ALIGN
    for bad in (dict(lr=-1.0), dict(beta1=1.0), dict(beta2=-0.1), dict(eps=0.0),
                dict(weight_decay=float("nan")), dict(lr=float("inf"))):
        h = Z.AdamW(**bad).c()
        assert step(hp=ctypes.byref(h)) == Z.ZERO_ERR_INVALID, bad
    assert "zero_step" in Z.zero_last_error()
    assert Z.zero_launch_count() == before


def test_unfused_calls_reject_bad_arguments_without_launching(L):
    plan = Z.zero_plan_partitions([64, 64], 2, "round_robin")
    good = 1 << 20
    p2 = _arr([good, good])
    hp = Z.AdamW().c()
    before = Z.zero_launch_count()
    assert L.zero_reduce_scatter(plan.handle, p2, 0, 0, p2, 0, 0, None) == Z.ZERO_ERR_INVALID
    assert L.zero_reduce_scatter(plan.handle, p2, 0, 0, _arr([good, 0]), 3, 0, None) == Z.ZERO_ERR_INVALID
    assert L.zero_adamw_shard_step(plan.handle, p2, p2, p2, p2, None, 0, ctypes.byref(hp), 0, 3,
                                   None) == Z.ZERO_ERR_INVALID
    assert L.zero_allgather(plan.handle, p2, 0, None, 3, None) == Z.ZERO_ERR_INVALID
    assert L.zero_allgather(plan.handle, p2, 0, good + 6, 3, None) == Z.ZERO_ERR_ALIGN
    assert L.zero_init_shards(None, good, 0, p2, p2, p2, 3, None) == Z.ZERO_ERR_INVALID
    assert L.zero_init_shards(plan.handle, good, 3, p2, p2, p2, 3, None) == Z.ZERO_ERR_INVALID
    assert Z.zero_launch_count() == before


def test_binding_checks_sizes_before_the_library():
    torch = pytest.importorskip("torch")
    plan = Z.zero_plan_partitions([100, 28], 2, "flat", 16)
    cpu = torch.zeros(128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        Z.zero_step(plan, [cpu, cpu], "avg", [None] * 2, [None] * 2, [None] * 2, None, None,
                    Z.AdamW(), 1)


def test_binding_exports_every_declared_call(L):
    """The Python package exposes every C call under its C name."""
    import zero_sharded_optimizer_flatten_gb300 as pkg
    for n in _declared():
        assert hasattr(pkg, n), f"the binding lacks {n}"


def test_selftest_rejects_bad_limits(L):
    before = Z.zero_launch_count()
    for bad in (0, 999, 10**11):
        assert L.zero_selftest_wait_timeout(bad, None) == Z.ZERO_ERR_INVALID
    assert Z.zero_launch_count() == before


def test_more_calls_reject_bad_arguments_without_launching(L):
    """The range reduction, the ZeRO-3 pass, the offload steps and the
    reduced mixed-precision step refuse bad arguments with the documented
    status before any CUDA call (this host has no GPU), and launch nothing."""
    plan = Z.zero_plan_partitions([100, 28], 2, "flat", 16)     # padded 128, 2 shards of 64
    good = 1 << 20
    p2 = _arr([good, good])
    hp = Z.AdamW().c()
    cfg = Z.AmpConfig().c()
    before = Z.zero_launch_count()
    # a flat range outside [0, padded]
    for lo, hi in ((-1, 10), (10, 5), (0, 129)):
        assert L.zero_reduce_scatter_range(plan.handle, p2, 1, 1, p2, 3, lo, hi,
                                           None) == Z.ZERO_ERR_INVALID
    assert "range" in Z.zero_last_error()
    # the ZeRO-3 pass: no layer, no or too many buffers, a NULL or misaligned buffer
    layer = Z._LayerC(p2, p2, p2, p2, p2)
    one = (Z._LayerC * 1)(layer)
    assert L.zero_zero3_pass(plan.handle, one, 0, p2, 1, 1, 1, ctypes.byref(hp), 1, None,
                             None) == Z.ZERO_ERR_INVALID
    for nb in (0, 65):
        assert L.zero_zero3_pass(plan.handle, one, 1, p2, nb, 1, 1, ctypes.byref(hp), 1, None,
                                 None) == Z.ZERO_ERR_INVALID
    assert L.zero_zero3_pass(plan.handle, one, 1, _arr([0]), 1, 1, 1, ctypes.byref(hp), 1, None,
                             None) == Z.ZERO_ERR_INVALID
    assert L.zero_zero3_pass(plan.handle, one, 1, _arr([good + 2]), 1, 1, 1, ctypes.byref(hp),
                             1, None, None) == Z.ZERO_ERR_ALIGN

    # the offload steps: a bad op, step 0, a misaligned gathered buffer, no
    # 16-bit shards, too many chunks
    def offload(op=1, step=1, o16=p2, full=good):
        return L.zero_offload_step(plan.handle, p2, 1, op, p2, p2, p2, p2, o16, full,
                                   ctypes.byref(hp), step, 3, 0, 2, None)
    assert offload(op=7) == Z.ZERO_ERR_INVALID
    assert offload(step=0) == Z.ZERO_ERR_INVALID
    assert offload(full=good + 2) == Z.ZERO_ERR_ALIGN
    assert offload(o16=None) == Z.ZERO_ERR_INVALID
    big = Z.zero_plan_partitions([5000], 2, "flat", 16)       # 5024 chunks of 1 element
    assert L.zero_offload_step(big.handle, p2, 1, 1, p2, p2, p2, p2, p2, good, ctypes.byref(hp),
                               1, 3, 1, 2, None) == Z.ZERO_ERR_INVALID
    assert "chunks" in Z.zero_last_error()
    assert L.zero_offload_step_amp(big.handle, p2, 1, 1, p2, p2, p2, p2, p2, good,
                                   ctypes.byref(hp), ctypes.byref(cfg), good, good, 1 << 20, 3, 0,
                                   1, 2, None) == Z.ZERO_ERR_INVALID
    assert "chunks" in Z.zero_last_error()
    # the reduced mixed-precision step with a workspace that is too small
    need = Z.zero_amp_workspace_bytes(plan)
    assert L.zero_step_amp_reduced(plan.handle, 1, p2, p2, p2, p2, good, None, ctypes.byref(hp),
                                   ctypes.byref(cfg), good, good, need - 16, 3, 0,
                                   None) == Z.ZERO_ERR_INVALID
    assert "workspace" in Z.zero_last_error()
    assert Z.zero_launch_count() == before
