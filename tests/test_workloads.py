"""The seeded input generators: any sub-range drawn alone equals the same
range of a whole draw (the sampled full-size parity checks rely on it), the
tail padding is zero, and the five groups have the published sizes."""
import numpy as np
import torch

from zero_sharded_optimizer_flatten_gb300 import workloads as W


def test_subranges_match_the_whole_draw():
    w = W.small((W.CHUNK + 1234, 77, 3 * W.CHUNK // 2), 3, mode="flat", align=16, dtype="bf16",
                outlier_frac=0.01)
    L = w.phi + 50                    # a buffer with 50 elements of tail padding
    whole = W.grads16(w, 2, 1, "cpu", 0, L)
    rng = np.random.default_rng(0)
    for _ in range(8):
        lo = int(rng.integers(0, L - 1))
        hi = int(rng.integers(lo + 1, min(L, lo + 2 * W.CHUNK) + 1))
        part = W.grads16(w, 2, 1, "cpu", lo, hi)
        assert torch.equal(part, whole[lo:hi])
    assert not whole[w.phi:].any()


def test_draws_depend_on_step_rank_layer_kind():
    w = W.small((5000,), 2, dtype="fp16")
    n = w.phi
    a = W.grads16(w, 1, 0, "cpu", 0, n)
    assert not torch.equal(a, W.grads16(w, 2, 0, "cpu", 0, n))
    assert not torch.equal(a, W.grads16(w, 1, 1, "cpu", 0, n))
    assert not torch.equal(a, W.grads16(w, 1, 0, "cpu", 0, n, layer=1))
    assert not torch.equal(W.params16(w, "cpu", n), W.params16(w, "cpu", n, layer=1))
    assert torch.equal(a, W.grads16(w, 1, 0, "cpu", 0, n))        # reproducible


def test_scale_multiplies_before_rounding():
    w = W.small((5000,), 1, dtype="fp16", grad_sigma=1.0)
    n = w.phi
    big = W.grads16(w, 1, 0, "cpu", 0, n, scale=1e5).float()
    assert torch.isinf(big).any()                               # fp16 overflow appears
    assert torch.equal(W.grads16(w, 1, 0, "cpu", 0, n, scale=1.0),
                       W.grads16(w, 1, 0, "cpu", 0, n))


def test_group_sizes():
    sizes = {k: (w.phi, len(w.numel)) for k, w in W.WORKLOADS.items()}
    assert sizes["tiny_mlp"] == (1053706, 10)
    assert sizes["bert_base"] == (109482240, 199)
    assert sizes["toy_rr"] == (100734986, 50)
    assert sizes["llama7b_rank0"] == (6738415616, 291)
    assert sizes["llama13b_layer"] == (212336640, 3)
    assert sizes["llama13b_full_layer"] == (317204480, 9)
