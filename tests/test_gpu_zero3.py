"""The ZeRO-3 layer stream (zero_zero3_pass): gathers on one stream run ahead
of the fused steps on another.  Results must equal the oracle's layer pass
(per layer: gather the 16-bit shards into the layer buffer, then the step
writing each rank's shard) and the serial pass of the already-tested pieces
(zero_allgather then zero_step, layer by layer)."""
import gc

import numpy as np
import pytest
import torch

import oracle
from tests._harness import (assert_16_close, assert_fp32_close, dt_code, f32, hp_oracle,
                            mode_code, op_code, u16)
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


def _layers(w, plan, n_layers):
    out = []
    for layer in range(n_layers):
        p16 = W.params16(w, "cuda", plan.padded, layer=layer)
        S = [plan.shard_len(r) for r in range(w.n_ranks)]
        shards = []
        for r in range(w.n_ranks):       # rank r's 16-bit shard: its segments of p16
            sh = torch.empty(S[r], dtype=w.torch_dtype, device="cuda")
            for k, toff, foff, soff, ln in plan.segments(r):
                sh[soff:soff + ln] = p16[foff:foff + ln]
            shards.append(sh)
        L = {"grads": [W.grads16(w, 1, q, "cuda", 0, plan.padded, layer=layer)
                       for q in range(w.n_ranks)],
             "shards16": shards,
             "master": [torch.empty(n, dtype=torch.float32, device="cuda") for n in S]}
        L["m"] = [torch.empty_like(x) for x in L["master"]]
        L["v"] = [torch.empty_like(x) for x in L["master"]]
        Z.zero_init_shards(plan, p16, L["master"], L["m"], L["v"])
        L["p16"] = u16(p16)
        out.append(L)
    return out


def _oracle_layer(w, L):
    """The oracle's copy of one layer: master = the 16-bit partition widened,
    m = v = 0, the 16-bit shards and the gradient replicas as drawn."""
    o = {"master": [], "m": [], "v": [], "shards16": [u16(x) for x in L["shards16"]],
         "grads": [u16(x) for x in L["grads"]]}
    for r in range(w.n_ranks):
        seg = oracle.segments(list(w.numel), w.n_ranks, mode_code(w), w.align, r)
        S = int(seg[:, 4].sum()) if len(seg) else 0
        mst = np.zeros(S, np.float32)
        for k, toff, foff, soff, ln in seg:
            mst[soff:soff + ln] = oracle.to_f32(L["p16"][foff:foff + ln], dt_code(w))
        o["master"].append(mst)
        o["m"].append(np.zeros(S, np.float32))
        o["v"].append(np.zeros(S, np.float32))
    return o


ZERO3_LAYOUTS = {
    "flat_bf16_N4": dict(numel=(30000, 37, 4096, 3, 129), N=4, mode="flat", align=16,
                         dtype="bf16", op="avg"),
    "rr_fp16_N3_sum": dict(numel=(30000, 37, 4096, 3, 129, 777), N=3, mode="round_robin",
                           align=1, dtype="fp16", op="sum"),
}


@pytest.mark.parametrize("layout", sorted(ZERO3_LAYOUTS))
@pytest.mark.parametrize("n_bufs,two_streams", [(1, False), (1, True), (2, True), (3, True)])
def test_zero3_pass_equals_oracle_and_serial_pieces(n_bufs, two_streams, layout):
    cfg = ZERO3_LAYOUTS[layout]
    N = cfg["N"]
    w = W.small(cfg["numel"], N, mode=cfg["mode"], align=cfg["align"], dtype=cfg["dtype"],
                op=cfg["op"])
    plan = Z.zero_plan_partitions(list(w.numel), N, w.mode, w.align)
    n_layers = 5
    ref = _layers(w, plan, n_layers)
    got = _layers(w, plan, n_layers)
    orc = [_oracle_layer(w, L) for L in got]
    o_bufs = [np.zeros(plan.padded, np.uint16) for _ in range(n_layers)]
    ref_bufs = [torch.empty(plan.padded, dtype=w.torch_dtype, device="cuda")
                for _ in range(n_layers)]
    bufs = [torch.full((plan.padded,), 3.0, dtype=w.torch_dtype, device="cuda")
            for _ in range(n_bufs)]
    gather = torch.cuda.Stream() if two_streams else None
    passer = Z.Zero3Pass(plan, got, bufs, w.op, HP)
    hp = hp_oracle(HP)
    md, dt, op = mode_code(w), dt_code(w), op_code(w)
    after_step1 = None
    for t in (1, 2):
        for layer in range(n_layers):
            L = ref[layer]
            Z.zero_allgather(plan, L["shards16"], ref_bufs[layer])
            Z.zero_step(plan, L["grads"], w.op, L["master"], L["m"], L["v"], None,
                        L["shards16"], HP, t)
            # the oracle's layer pass: gather, then the step writing the shards
            o = orc[layer]
            oracle.allgather(list(w.numel), N, md, w.align, o["shards16"], o_bufs[layer])
            oracle.step(list(w.numel), N, md, w.align, dt, op, o["grads"], o["master"], o["m"],
                        o["v"], None, o["shards16"], hp, t)
        passer(t, gather_stream=gather)
        if t == 1:
            torch.cuda.synchronize()
            after_step1 = [[u16(x) for x in L["shards16"]] for L in got]
    torch.cuda.synchronize()
    for layer in range(n_layers):
        o = orc[layer]
        for r in range(N):
            for key in ("master", "m", "v", "shards16"):
                assert torch.equal(got[layer][key][r], ref[layer][key][r]), (layer, key, r)
            what = f"{layout} layer {layer} rank {r}"
            assert_fp32_close(f32(got[layer]["master"][r]), o["master"][r], what + " master")
            assert_fp32_close(f32(got[layer]["m"][r]), o["m"][r], what + " m")
            assert_fp32_close(f32(got[layer]["v"][r]), o["v"][r], what + " v")
            assert_16_close(u16(got[layer]["shards16"][r]), o["shards16"][r], what + " shard16",
                            dtype_code=dt)
    # each buffer holds the last gather that used it (of step 2): the oracle's
    # gather of the shards the pass wrote at step 1, bit for bit, and the
    # oracle's own layer buffer within the 16-bit bar
    for b in range(n_bufs):
        last = max(l for l in range(n_layers) if l % n_bufs == b)
        assert torch.equal(bufs[b], ref_bufs[last])
        want = np.zeros(plan.padded, np.uint16)
        oracle.allgather(list(w.numel), N, md, w.align, after_step1[last], want)
        assert np.array_equal(u16(bufs[b]), want), f"buffer {b}"
        assert_16_close(u16(bufs[b]), o_bufs[last], f"buffer {b}", dtype_code=dt)


def test_zero3_pass_rejects_a_bad_layer_before_launching():
    w = W.small((4096,), 2, mode="flat", align=16, dtype="bf16", op="avg")
    plan = Z.zero_plan_partitions(list(w.numel), 2, "flat", 16)
    layers = _layers(w, plan, 3)
    buf = torch.empty(plan.padded, dtype=w.torch_dtype, device="cuda")
    passer = Z.Zero3Pass(plan, layers, [buf], "avg", HP)
    # corrupt layer 2's master pointer for rank 1 to a misaligned address
    base = layers[2]["master"][1].data_ptr()
    passer._arrays[2][1][1] = base + 4
    before = Z.zero_launch_count()
    with pytest.raises(Z.ZeroError) as e:
        passer(1)
    assert e.value.status == Z.ZERO_ERR_ALIGN and "layer 2" in str(e.value)
    assert Z.zero_launch_count() == before


@pytest.mark.parametrize("two_streams", [False, True])
def test_zero3_pass_with_layer_state_in_host_memory(two_streams):
    """ZeRO-3 with the layers' state offloaded: every layer's 16-bit shards
    and fp32 master/m/v live in pinned host memory (the gradient replicas and
    the layer buffers stay in HBM); the gathers read the shards and the steps
    update the state across the host link.  Bit for bit the device-resident
    pass."""
    cfg = ZERO3_LAYOUTS["flat_bf16_N4"]
    N = cfg["N"]
    w = W.small(cfg["numel"], N, mode=cfg["mode"], align=cfg["align"], dtype=cfg["dtype"],
                op=cfg["op"])
    plan = Z.zero_plan_partitions(list(w.numel), N, w.mode, w.align)
    n_layers = 4
    dev = _layers(w, plan, n_layers)
    host = _layers(w, plan, n_layers)
    for L in host:
        for key in ("shards16", "master", "m", "v"):
            L[key] = [x.cpu().pin_memory() for x in L[key]]
    dbufs = [torch.zeros(plan.padded, dtype=w.torch_dtype, device="cuda") for _ in range(2)]
    hbufs = [torch.zeros(plan.padded, dtype=w.torch_dtype, device="cuda") for _ in range(2)]
    gather = torch.cuda.Stream() if two_streams else None
    pass_dev = Z.Zero3Pass(plan, dev, dbufs, w.op, HP)
    pass_host = Z.Zero3Pass(plan, host, hbufs, w.op, HP)
    for t in (1, 2, 3):
        pass_dev(t, gather_stream=gather)
        pass_host(t, gather_stream=gather)
    torch.cuda.synchronize()
    for layer in range(n_layers):
        for r in range(N):
            for key in ("master", "m", "v", "shards16"):
                assert torch.equal(host[layer][key][r], dev[layer][key][r].cpu()), (layer, key)
    for b in range(2):
        assert torch.equal(hbufs[b], dbufs[b])
