"""A ZeRO data-parallel engine over N virtual ranks on one GPU.

It wires a model's backward pass into the library's calls the way
"DeepSpeed ZeRO-2 ... DeepSpeedZeroOptimizer" (discosf.com) §2.1 and §4.1-§4.4
describe the optimizer doing it:

* the parameters are flattened into one 16-bit buffer (and become views of
  it), which the plan partitions across the ranks;
* every virtual rank q owns one flat gradient replica (contiguous gradients);
  a post-accumulate-grad hook copies each parameter's gradient into rank q's
  replica and releases ``param.grad`` (the ZeRO-2 release of gradients);
* the replicas are cut into buckets of ``bucket_elems`` flat elements (the
  IPG bucket, reduce_bucket_size); as soon as every rank has filled a bucket,
  its reduce-scatter is launched -- on a side stream when ``overlap_comm`` so
  it runs while the backward pass goes on;
* ``step()`` waits for the reductions, runs AdamW on every rank's fp32 shard,
  casts to 16 bits and all-gathers into the flat buffer, so the model's
  parameters hold the new values.

With ``amp`` (an ``AmpConfig``) the engine is the fp16 ZeRO-2 loop of the
pages' ds_config (fp16 loss_scale 0 = dynamic, loss_scale_window,
hysteresis, min_loss_scale, gradient_clipping): ``backward`` multiplies each
rank's loss by the current loss scale, read on the device from the state
buffer (no host synchronisation); each bucket's reduction also writes its
tiles' sums of squares (``zero_reduce_scatter_bucket_amp``), and ``step()``
runs the rest of the mixed-precision step on the reduced shards (overflow
skip, scale update, clipping, AdamW, cast, gather;
``zero_step_amp_reduced``), bit-identical to ``zero_step_amp`` on the
replicas with the same bucket size.

With ``offload`` the fp32 optimizer state lives in pinned host memory, as
the pages' ds_config ``offload_optimizer: {device: cpu, pin_memory: true}``
asks ("DeepSpeed ZeRO-2 ..." §4.5).  ``offload="cpu"`` is that form: the
bucket reductions write the fp32 gradient shards into pinned host memory
across the host link, ``step()`` runs AdamW + cast on host threads and
all-gathers the host 16-bit shards, chunk by chunk so that the gathers
overlap the update (``zero_offload_step`` on the reduced shards; with ``amp`` the device
still takes the decision and the host applies it,
``zero_offload_step_amp``).  ``offload="host_state"`` keeps the update on
the GPU, whose kernels read and write the host-resident master/m/v across
NVLink-C2C (no host synchronisation).  Both give the device engine's results
bit for bit.  ``host_threads`` sets the CPU optimizer's threads (0: every
hardware thread but one).

The arithmetic is the library's (no compute happens here); this module only
does bookkeeping and launches.
"""
from __future__ import annotations

from typing import Iterable, List, Optional

import torch

from . import zero as Z


class ZeroEngine:
    def __init__(self, params: Iterable[torch.nn.Parameter], n_ranks: int, *, mode="flat",
                 align: int = 16, op: str = "avg", hparams: Optional[Z.AdamW] = None,
                 bucket_elems: int = 50_000_000, overlap_comm: bool = True,
                 amp: Optional[Z.AmpConfig] = None, offload: Optional[str] = None,
                 host_threads: int = 0):
        self.params: List[torch.nn.Parameter] = list(params)
        if not self.params:
            raise ValueError("no parameters")
        dt = self.params[0].dtype
        dev = self.params[0].device
        if dt not in (torch.float16, torch.bfloat16):
            raise TypeError("parameters must be float16 or bfloat16 (the 16-bit model copy)")
        for p in self.params:
            if p.dtype != dt or p.device != dev or not p.is_cuda:
                raise ValueError("all parameters must share one 16-bit dtype and one CUDA device")
        if offload not in (None, "cpu", "host_state"):
            raise ValueError("offload must be None, 'cpu' or 'host_state'")
        self.offload, self.host_threads = offload, host_threads
        self.n_ranks, self.op = n_ranks, op
        self.hp = hparams or Z.AdamW()
        self.numel = [p.numel() for p in self.params]
        self.plan = plan = Z.zero_plan_partitions(self.numel, n_ranks, mode, align)
        P, phi = plan.padded, plan.phi
        # flat 16-bit parameters; the model's parameters become views of it
        self.flat16 = torch.zeros(P, dtype=dt, device=dev)
        self.offsets, off = [], 0
        with torch.no_grad():
            for p, n in zip(self.params, self.numel):
                self.flat16[off:off + n].copy_(p.reshape(-1))
                p.data = self.flat16[off:off + n].view_as(p)
                self.offsets.append(off)
                off += n
        # per-rank gradient replicas, fp32 gradient shards, optimizer state
        self.grads = [torch.zeros(P, dtype=dt, device=dev) for _ in range(n_ranks)]
        S = [plan.shard_len(r) for r in range(n_ranks)]

        def shard_buf(n, dtype, on_host):
            if on_host:
                return torch.zeros(n, dtype=dtype, pin_memory=True)
            return torch.zeros(n, dtype=dtype, device=dev)
        host = offload == "cpu"
        self.grad_shards = [shard_buf(n, torch.float32, host) for n in S]
        self.master = [shard_buf(n, torch.float32, offload is not None) for n in S]
        self.m = [shard_buf(n, torch.float32, offload is not None) for n in S]
        self.v = [shard_buf(n, torch.float32, offload is not None) for n in S]
        self.shard16 = [shard_buf(n, dt, host) for n in S]
        # master = the 16-bit values widened, m = v = 0 (the kernel writes
        # host-resident state across the link as well)
        Z.zero_init_shards(plan, self.flat16, self.master, self.m, self.v)
        # buckets over the flat index space; the tail padding needs no filling
        B = bucket_elems if bucket_elems > 0 else P
        self.bucket_elems = B
        self.buckets = [(lo, min(lo + B, P)) for lo in range(0, P, B)]
        self._need = [max(0, min(hi, phi) - min(lo, phi)) for lo, hi in self.buckets]
        self._tensor_buckets = []
        for k, (o, n) in enumerate(zip(self.offsets, self.numel)):
            parts = []
            for b in range(o // B, (o + n - 1) // B + 1 if n else o // B):
                lo, hi = self.buckets[b]
                cnt = min(hi, o + n) - max(lo, o)
                if cnt > 0:
                    parts.append((b, cnt))
            self._tensor_buckets.append(parts)
        self.reduction_stream = torch.cuda.Stream(dev) if overlap_comm else None
        self._reduce = Z.ReduceScatterRange(plan, self.grads, op, self.grad_shards)
        # mixed-precision controls: device state, its loss scale as a tensor
        # view (the state's first field), the step's workspace; each bucket's
        # reduction also writes its tiles' sums of squares into the workspace,
        # so the step reads the gradient shards once (for the update)
        self.amp = amp
        if amp is not None:
            self.amp_state = Z.amp_state_tensor(dev)
            Z.zero_amp_init(self.amp_state, amp)
            self._scale = self.amp_state[:8].view(torch.float64)[0]
            self._workspace = torch.empty(max(16, Z.zero_amp_workspace_bytes(plan,
                                                                               bucket_elems=B)),
                                          dtype=torch.uint8, device=dev)
            self._reduce_amp = Z.ReduceScatterBucketAmp(plan, self.grads, op, self.grad_shards,
                                                        self.hp, self.amp_state, self._workspace,
                                                        bucket_elems=B)
        self.step_count = 0
        self.launched_during_backward = 0
        self._current: Optional[int] = None
        self._reset()
        self._hooks = [p.register_post_accumulate_grad_hook(self._hook(k))
                       for k, p in enumerate(self.params)]

    # ------------------------------------------------------------------
    def _reset(self):
        nb = len(self.buckets)
        self._filled = [[0] * nb for _ in range(self.n_ranks)]
        self._ranks_done = [0] * nb
        self._launched = [False] * nb
        self._seen = [False] * self.n_ranks

    def _hook(self, k: int):
        def hook(p: torch.nn.Parameter):
            q = self._current
            if q is None or p.grad is None:
                return  # a backward pass outside backward(): leave .grad alone
            o, n = self.offsets[k], self.numel[k]
            self.grads[q][o:o + n].copy_(p.grad.reshape(-1))
            p.grad = None
            for b, cnt in self._tensor_buckets[k]:
                self._filled[q][b] += cnt
                if self._filled[q][b] == self._need[b]:
                    self._ranks_done[b] += 1
                    if self._ranks_done[b] == self.n_ranks:
                        self._launch(b)
                        self.launched_during_backward += 1
        return hook

    def _launch(self, b: int):
        lo, hi = self.buckets[b]
        stream = None
        if self.reduction_stream is not None:
            # the replica copies were queued on the current stream
            self.reduction_stream.wait_stream(torch.cuda.current_stream())
            stream = self.reduction_stream
        if self.amp is not None:
            self._reduce_amp(b, stream=stream)
        else:
            self._reduce(lo, hi, stream=stream)
        self._launched[b] = True

    # ------------------------------------------------------------------
    def backward(self, loss: torch.Tensor, rank: int):
        """loss.backward() for virtual rank `rank` (its micro-batch)."""
        if not 0 <= rank < self.n_ranks:
            raise ValueError(f"rank {rank} out of range")
        if self._seen[rank]:
            raise RuntimeError(f"rank {rank} already ran backward in this iteration")
        self._current = rank
        try:
            if self.amp is not None:
                loss = loss * self._scale.to(loss.dtype)
            loss.backward()
        finally:
            self._current = None
        self._seen[rank] = True
        for b, need in enumerate(self._need):
            if need == 0 and not self._launched[b] and all(self._seen):
                self._launch(b)  # buckets of padding only

    def step(self):
        """Wait for the reductions, then AdamW + cast + all-gather."""
        if not all(self._seen):
            missing = [q for q in range(self.n_ranks) if not self._seen[q]]
            raise RuntimeError(f"ranks {missing} did not run backward in this iteration")
        for b, done in enumerate(self._launched):
            if not done:
                raise RuntimeError(f"bucket {b} was not filled by every rank (a parameter "
                                   "received no gradient?)")
        if self.reduction_stream is not None:
            torch.cuda.current_stream().wait_stream(self.reduction_stream)
        self.step_count += 1
        if self.amp is not None and self.offload == "cpu":
            # the device decides (skip, loss scale, clipping); the host reads
            # the decision and updates; the gathers overlap the update
            Z.zero_offload_step_amp(self.plan, None, self.op, self.grad_shards, self.master,
                                    self.m, self.v, self.shard16, self.flat16, self.hp, self.amp,
                                    self.amp_state, self._workspace,
                                    bucket_elems=self.bucket_elems,
                                    n_threads=self.host_threads)
        elif self.amp is not None:
            # the step count that AdamW uses lives in the device state (skipped
            # steps do not count)
            Z.zero_step_amp_reduced(self.plan, self.grad_shards, self.master, self.m, self.v,
                                    self.flat16, None, self.hp, self.amp, self.amp_state,
                                    self._workspace, bucket_elems=self.bucket_elems)
        elif self.offload == "cpu":
            # the gradient shards are reduced already: the host update waits
            # for the stream, and each chunk's gather overlaps the next
            # chunk's update
            Z.zero_offload_step(self.plan, None, self.op, self.grad_shards, self.master, self.m,
                                self.v, self.shard16, self.flat16, self.hp, self.step_count,
                                n_threads=self.host_threads)
        else:
            Z.zero_adamw_shard_step(self.plan, self.master, self.m, self.v, self.grad_shards,
                                    self.shard16, self.hp, self.step_count)
            Z.zero_allgather(self.plan, self.shard16, self.flat16)
        self._reset()

    def state_dict(self) -> dict:
        """Host copies of everything a resumed run needs: the fp32 master, m
        and v of every rank, the 16-bit flat parameters, the step count and
        the mixed-precision state (the checkpoint of the optimizer; saving it
        is the caller's, e.g. torch.save)."""
        # host-resident state is written by the device (offload='host_state')
        # or read by its gathers: wait for every stream before copying
        torch.cuda.synchronize(self.flat16.device)

        def host(xs):
            return [x.detach().cpu().clone() for x in xs]
        sd = {"numel": list(self.numel), "n_ranks": self.n_ranks, "mode": self.plan.mode,
              "align": self.plan.align, "step_count": self.step_count,
              "master": host(self.master), "m": host(self.m), "v": host(self.v),
              "flat16": self.flat16.detach().cpu().clone()}
        if self.amp is not None:
            sd["amp_state"] = self.amp_state.detach().cpu().clone()
        return sd

    def load_state_dict(self, sd: dict):
        """Restore a state_dict() of an engine over the same parameter group:
        the model's parameters (views of the flat buffer) and the optimizer
        state take the saved values, so training continues bit for bit."""
        same = (list(sd["numel"]) == list(self.numel) and sd["n_ranks"] == self.n_ranks
                and sd["mode"] == self.plan.mode and sd["align"] == self.plan.align)
        if not same:
            raise ValueError("the checkpoint was taken over another parameter group or plan")
        if ("amp_state" in sd) != (self.amp is not None):
            raise ValueError("the checkpoint and the engine disagree on amp")
        torch.cuda.synchronize(self.flat16.device)   # no kernel still uses the old state
        with torch.no_grad():
            for key in ("master", "m", "v"):
                for dst, src in zip(getattr(self, key), sd[key]):
                    if dst.shape != src.shape:
                        raise ValueError(f"{key}: shard of {tuple(src.shape)}, expected "
                                         f"{tuple(dst.shape)}")
                    dst.copy_(src)
            self.flat16.copy_(sd["flat16"])
            if self.amp is not None:
                self.amp_state.copy_(sd["amp_state"])
        self.step_count = int(sd["step_count"])
        self._reset()

    def amp_status(self) -> "Z.AmpState":
        """The mixed-precision state (loss scale, last norm, steps taken and
        skipped); copying it to the host synchronises with the stream."""
        if self.amp is None:
            raise RuntimeError("the engine was built without amp")
        return Z.read_amp_state(self.amp_state)

    def remove_hooks(self):
        for h in self._hooks:
            h.remove()
        self._hooks = []
