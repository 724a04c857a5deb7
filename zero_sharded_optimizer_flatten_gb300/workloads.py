"""Seeded synthetic workloads for the ZeRO sharded optimizer step.

This module describes the five parameter groups the step is exercised on and
draws their random inputs.  It holds none of the step's arithmetic (no
partitioning, reduction, AdamW or rounding of results): it only lists tensor
shapes and fills buffers with seeded normal samples, so the CPU oracle and the
CUDA path can both be fed from it.

Tensor lists are in ``named_parameters()`` order, weight before bias, for
torch ``nn.Linear(in, out)`` (weight shape (out, in)).  Sources for the
shapes: the ToyModel of "ZeRO ... 实操" (wmrh.cn) §3.1 (hidden 1024, 12
layers of Linear(1024, 4096) + Linear(4096, 1024), classifier
Linear(1024, 10)); BERT-base and LLaMA sizes as named in the same tutorial
(§2.1 "BERT-base 110M", §1 "LLaMA 7B").  The vocabulary (32000), BERT's
position/type/pooler tensors and the LLaMA-13B MLP-only layer are readings
chosen to reproduce the parameter counts "110M", "6.74B" and "~212M".

Random draws: the flat index space of each buffer is cut into fixed chunks of
``CHUNK`` elements, and chunk c of (workload, kind, step, rank) is drawn from
its own ``torch.Generator`` seeded by a hash of that tuple.  Any sub-range can
therefore be regenerated alone (the sampled full-size parity checks rely on
it).  Streams differ between CPU and CUDA generators, so a run draws all its
inputs on one device and copies what the oracle needs to the host.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import List, Optional

import torch

CHUNK = 1 << 22


@dataclasses.dataclass(frozen=True)
class Workload:
    key: str
    title: str
    numel: tuple
    n_ranks: int
    mode: str           # "flat" or "round_robin"
    align: int          # alignment of the flat partition (elements); unused for round_robin
    dtype: str          # "fp16" or "bf16"
    op: str             # "sum" or "avg"
    param_sigma: float
    grad_sigma: float
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    steps: int = 3
    rank_mask: Optional[int] = None   # None: every rank
    bucket_elems: int = 0             # 0: one bucket
    layers: int = 1                   # ZeRO-3 layer streaming: layers per pass
    zero3: bool = False               # write each rank's 16-bit shard (next gather's source)
    seed: int = 0

    @property
    def phi(self) -> int:
        return int(sum(self.numel))

    @property
    def mask(self) -> int:
        return (1 << self.n_ranks) - 1 if self.rank_mask is None else self.rank_mask

    @property
    def torch_dtype(self):
        return torch.float16 if self.dtype == "fp16" else torch.bfloat16


def _linear(i, o):
    return [o * i, o]


def tiny_mlp_numel() -> List[int]:
    out = []
    for _ in range(2):
        out += _linear(256, 1024) + _linear(1024, 256)
    return out + _linear(256, 10)


def bert_base_numel(vocab=30522, hidden=768, ffn=3072, layers=12, max_pos=512, types=2):
    h = hidden
    out = [vocab * h, max_pos * h, types * h, h, h]           # embeddings + LayerNorm
    for _ in range(layers):
        out += _linear(h, h) + _linear(h, h) + _linear(h, h)      # query, key, value
        out += _linear(h, h)                                    # attention output dense
        out += [h, h]                                           # attention LayerNorm
        out += _linear(h, ffn) + _linear(ffn, h)                # intermediate, output
        out += [h, h]                                           # output LayerNorm
    out += _linear(h, h)                                        # pooler
    return out


def toy_model_numel(hidden=1024, layers=12, classes=10):
    out = []
    for _ in range(layers):
        out += _linear(hidden, 4 * hidden) + _linear(4 * hidden, hidden)
    return out + _linear(hidden, classes)


def llama_numel(vocab=32000, hidden=4096, ffn=11008, layers=32):
    h = hidden
    out = [vocab * h]
    for _ in range(layers):
        out += [h * h] * 4                 # q, k, v, o projections (no bias)
        out += [ffn * h, ffn * h, h * ffn]  # gate, up, down
        out += [h, h]                      # input / post-attention RMSNorm
    out += [h, vocab * h]                  # final norm, lm_head
    return out


def llama13b_mlp_numel(hidden=5120, ffn=13824):
    return [ffn * hidden, ffn * hidden, hidden * ffn]


def llama13b_layer_numel(hidden=5120, ffn=13824):
    """A whole LLaMA-13B decoder layer: q, k, v, o, gate, up, down, 2 norms."""
    h = hidden
    return [h * h] * 4 + [ffn * h, ffn * h, h * ffn] + [h, h]


WORKLOADS = {
    "tiny_mlp": Workload(
        "tiny_mlp", "tiny MLP 2x[Linear(256,1024)+Linear(1024,256)]+Linear(256,10), fp16, "
        "N=4 flat, A=16", tuple(tiny_mlp_numel()), 4, "flat", 16, "fp16", "avg", 0.02, 1e-2,
        steps=3, seed=1235),
    "bert_base": Workload(
        "bert_base", "BERT-base 110M flat group, bf16, N=8 flat, averaged",
        tuple(bert_base_numel()), 8, "flat", 16, "bf16", "avg", 0.02, 1e-3, steps=10,
        seed=1236),
    "toy_rr": Workload(
        "toy_rr", "ToyModel hidden 1024 x12 + Linear(1024,10), fp16, N=4 round-robin, summed, "
        "1% of gradient entries x100", tuple(toy_model_numel()), 4, "round_robin", 1, "fp16",
        "sum", 0.02, 1e-2, outlier_frac=0.01, outlier_scale=100.0, steps=3, seed=1237),
    "llama7b_rank0": Workload(
        "llama7b_rank0", "LLaMA-7B group (6.74B), N=8 flat, rank 0's 842M-element shard, bf16, "
        "averaged, 50M-element buckets", tuple(llama_numel()), 8, "flat", 16, "bf16", "avg",
        0.02, 1e-3, steps=3, rank_mask=1, bucket_elems=50_000_000, seed=1238),
    "llama13b_layer": Workload(
        "llama13b_layer", "ZeRO-3 pass over 40 LLaMA-13B MLP layers (212M each), N=8 flat, "
        "bf16, averaged", tuple(llama13b_mlp_numel()), 8, "flat", 16, "bf16", "avg", 0.02,
        1e-3, steps=1, layers=40, zero3=True, seed=1239),
    "llama13b_full_layer": Workload(
        "llama13b_full_layer", "ZeRO-3 pass over 40 whole LLaMA-13B decoder layers (317M each), "
        "N=8 flat, bf16, averaged", tuple(llama13b_layer_numel()), 8, "flat", 16, "bf16", "avg",
        0.02, 1e-3, steps=1, layers=40, zero3=True, seed=1240),
}


def _seed(*parts) -> int:
    h = hashlib.blake2b(repr(parts).encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def _chunk(w: Workload, kind: str, step: int, rank: int, c: int, n: int, sigma: float,
           device, scale: float = 1.0) -> torch.Tensor:
    gen = torch.Generator(device=device)
    gen.manual_seed(_seed(w.seed, kind, step, rank, c))
    x = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    x.mul_(sigma)
    if kind == "grad" and w.outlier_frac > 0:
        hit = torch.rand(n, generator=gen, device=device, dtype=torch.float32) < w.outlier_frac
        x = torch.where(hit, x * w.outlier_scale, x)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(w.torch_dtype)


def fill(w: Workload, kind: str, step: int, rank: int, lo: int, hi: int, out: torch.Tensor,
         layer: int = 0, scale: float = 1.0) -> torch.Tensor:
    """Write the seeded values of flat range [lo, hi) into ``out`` (length hi-lo).

    kind "param": the initial 16-bit parameters (sigma = param_sigma);
    kind "grad": rank `rank`'s gradient replica at `step` (sigma = grad_sigma),
    multiplied by `scale` (a loss scale the backward pass would carry) before
    the rounding to 16 bits, so large scales overflow to infinity.
    Elements at or beyond phi (the tail padding) are zero.
    """
    assert out.numel() == hi - lo and out.dtype == w.torch_dtype
    sigma = w.param_sigma if kind == "param" else w.grad_sigma
    dev = out.device
    real_hi = min(hi, w.phi)
    if real_hi < hi:
        out[max(real_hi, lo) - lo:].zero_()
    c = lo // CHUNK
    while c * CHUNK < real_hi:
        c0, c1 = c * CHUNK, min((c + 1) * CHUNK, w.phi)
        a, b = max(c0, lo), min(c1, real_hi)
        if a < b:
            vals = _chunk(w, kind, step, rank if kind == "grad" else -1, (layer, c), c1 - c0,
                          sigma, dev, scale)
            out[a - lo:b - lo].copy_(vals[a - c0:b - c0])
        c += 1
    return out


def params16(w: Workload, device, n: int, layer: int = 0) -> torch.Tensor:
    """The initial 16-bit parameters of flat range [0, n); n is the flat
    buffer length the caller's plan gives (tail padding included)."""
    return fill(w, "param", 0, 0, 0, n, torch.empty(n, dtype=w.torch_dtype, device=device), layer)


def grads16(w: Workload, step: int, rank: int, device, lo: int, hi: int, layer: int = 0,
            scale: float = 1.0) -> torch.Tensor:
    """Rank `rank`'s gradient replica at `step` over flat range [lo, hi)."""
    return fill(w, "grad", step, rank, lo, hi,
                torch.empty(hi - lo, dtype=w.torch_dtype, device=device), layer, scale)


def small(numel, n_ranks, mode="flat", align=16, dtype="fp16", op="avg", grad_sigma=1e-2,
          outlier_frac=0.0, seed=7, **kw) -> Workload:
    """An ad-hoc workload for tests (tiny groups, edge cases)."""
    return Workload("adhoc", "adhoc", tuple(int(x) for x in numel), n_ranks, mode, align, dtype,
                    op, 0.02, grad_sigma, outlier_frac=outlier_frac,
                    outlier_scale=100.0 if outlier_frac else 1.0, seed=seed, **kw)
