"""The ZeRO-3 layer stream (zero_zero3_pass): gathers on one stream run ahead
of the fused steps on another; results must equal the serial pass of the
already-tested pieces (zero_allgather then zero_step, layer by layer)."""
import gc

import pytest
import torch

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
        p16 = W.params16(w, "cuda", layer=layer)
        off = [plan.shards[r][0] for r in range(w.n_ranks)]
        S = [plan.shard_len(r) for r in range(w.n_ranks)]
        L = {"grads": [W.grads16(w, 1, q, "cuda", layer=layer) for q in range(w.n_ranks)],
             "shards16": [p16[off[r]:off[r] + S[r]].clone() for r in range(w.n_ranks)],
             "master": [torch.empty(n, dtype=torch.float32, device="cuda") for n in S]}
        L["m"] = [torch.empty_like(x) for x in L["master"]]
        L["v"] = [torch.empty_like(x) for x in L["master"]]
        Z.zero_init_shards(plan, p16, L["master"], L["m"], L["v"])
        out.append(L)
    return out


@pytest.mark.parametrize("n_bufs,two_streams", [(1, False), (1, True), (2, True), (3, True)])
def test_zero3_pass_equals_serial_pieces(n_bufs, two_streams):
    w = W.small((30000, 37, 4096, 3, 129), 4, mode="flat", align=16, dtype="bf16", op="avg")
    plan = Z.zero_plan_partitions(list(w.numel), 4, "flat", 16)
    n_layers = 5
    ref = _layers(w, plan, n_layers)
    got = _layers(w, plan, n_layers)
    ref_bufs = [torch.empty(plan.padded, dtype=w.torch_dtype, device="cuda")
                for _ in range(n_layers)]
    bufs = [torch.full((plan.padded,), 3.0, dtype=w.torch_dtype, device="cuda")
            for _ in range(n_bufs)]
    gather = torch.cuda.Stream() if two_streams else None
    passer = Z.Zero3Pass(plan, got, bufs, "avg", HP)
    for t in (1, 2):
        for layer in range(n_layers):
            L = ref[layer]
            Z.zero_allgather(plan, L["shards16"], ref_bufs[layer])
            Z.zero_step(plan, L["grads"], "avg", L["master"], L["m"], L["v"], None,
                        L["shards16"], HP, t)
        passer(t, gather_stream=gather)
    torch.cuda.synchronize()
    for layer in range(n_layers):
        for r in range(4):
            for key in ("master", "m", "v", "shards16"):
                assert torch.equal(got[layer][key][r], ref[layer][key][r]), (layer, key, r)
    # each buffer holds the last gather that used it (of step 2)
    for b in range(n_bufs):
        last = max(l for l in range(n_layers) if l % n_bufs == b)
        assert torch.equal(bufs[b], ref_bufs[last])


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
