"""Python binding of the C ABI in include/zero.h (ctypes; argument marshalling only).

Every function keeps the C name and forwards to libzero.so.  Tensors are
torch tensors on the GPU or in pinned host memory (which the kernels read and
write across the host link), or raw integer addresses; the binding only
checks dtypes, devices, contiguity and sizes against the plan, turns them into
pointer arrays and passes the current CUDA stream.  There is no fallback: if
libzero.so is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzero.so")

ZERO_OK, ZERO_ERR_INVALID, ZERO_ERR_ALIGN, ZERO_ERR_CUDA, ZERO_ERR_OOM = 0, 1, 2, 3, 4
ZERO_ERR_TIMEOUT, ZERO_ERR_UNSUPPORTED = 5, 6
ZERO_FP16, ZERO_BF16 = 0, 1
ZERO_PART_FLAT, ZERO_PART_ROUND_ROBIN = 0, 1
ZERO_REDUCE_SUM, ZERO_REDUCE_AVG = 0, 1

_MODES = {"flat": ZERO_PART_FLAT, "round_robin": ZERO_PART_ROUND_ROBIN}
_OPS = {"sum": ZERO_REDUCE_SUM, "avg": ZERO_REDUCE_AVG}

_lock = threading.Lock()
_lib = None


class ZeroError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[status {status}] {message}")
        self.status = status


class AdamWHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("weight_decay", ctypes.c_double)]


@dataclasses.dataclass
class AdamW:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01

    def c(self) -> AdamWHparams:
        return AdamWHparams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay)


def lib():
    """Load libzero.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; "
                    "g.build()'` (needs nvcc); there is no fallback implementation")
            L = ctypes.CDLL(LIB_PATH)
            i64, i32, u64, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_void_p
            i64p, i32p = ctypes.POINTER(i64), ctypes.POINTER(i32)
            vpp = ctypes.POINTER(vp)
            hp = ctypes.POINTER(AdamWHparams)
            sig = {
                "zero_plan_partitions": [i64p, i32, i32, ctypes.c_int, i32,
                                         ctypes.POINTER(vp)],
                "zero_plan_total": [vp, i64p, i64p],
                "zero_plan_info": [vp, i32p, i32p, i32p, i32p],
                "zero_plan_shard": [vp, i32, i64p, i64p],
                "zero_plan_segments": [vp, i32, i64p, i64p, i64p, i64p, i64p, i64, i64p],
                "zero_plan_describe": [vp, ctypes.c_char_p, i64],
                "zero_memory_bytes": [i32, i64, i32, i64p, i64p],
                "zero_init_shards": [vp, vp, ctypes.c_int, vpp, vpp, vpp, u64, vp],
                "zero_reduce_scatter": [vp, vpp, ctypes.c_int, ctypes.c_int, vpp, u64, i64, vp],
                "zero_adamw_shard_step": [vp, vpp, vpp, vpp, vpp, vpp, ctypes.c_int, hp, i64,
                                          u64, vp],
                "zero_allgather": [vp, vpp, ctypes.c_int, vp, u64, vp],
                "zero_step": [vp, vpp, ctypes.c_int, ctypes.c_int, vpp, vpp, vpp, vp, vpp, hp,
                              i64, u64, i64, vp],
                "zero_floor_probe": [vp, i32, vpp, ctypes.c_int, vpp, vpp, vpp, vp, u64, i64, vp],
                "zero_sync": [vp],
                "zero_selftest_wait_timeout": [i64, vp],
                "zero_reduce_scatter_range": [vp, vpp, ctypes.c_int, ctypes.c_int, vpp, u64, i64,
                                              i64, vp],
                "zero_cpu_adamw_shard_step": [vp, vpp, vpp, vpp, vpp, vpp, ctypes.c_int, hp, i64,
                                              u64, i32],
                "zero_offload_step": [vp, vpp, ctypes.c_int, ctypes.c_int, vpp, vpp, vpp, vpp,
                                      vpp, vp, hp, i64, u64, i64, i32, vp],
                "zero_offload_step_amp": [vp, vpp, ctypes.c_int, ctypes.c_int, vpp, vpp, vpp,
                                          vpp, vpp, vp, hp, ctypes.POINTER(AmpConfigC), vp, vp,
                                          i64, u64, i64, i64, i32, vp],
                "zero_amp_init": [vp, ctypes.POINTER(AmpConfigC), vp],
                "zero_amp_workspace_bytes": [vp, u64, i64, i64p],
                "zero_step_amp": [vp, vpp, ctypes.c_int, ctypes.c_int, vpp, vpp, vpp, vpp, vp,
                                  vpp, hp, ctypes.POINTER(AmpConfigC), vp, vp, i64, u64, i64, vp],
                "zero_step_amp_shards": [vp, ctypes.c_int, vpp, vpp, vpp, vpp, vp, vpp, hp,
                                         ctypes.POINTER(AmpConfigC), vp, vp, i64, u64, i64, vp],
                "zero_step_amp_reduced": [vp, ctypes.c_int, vpp, vpp, vpp, vpp, vp, vpp, hp,
                                          ctypes.POINTER(AmpConfigC), vp, vp, i64, u64, i64, vp],
                "zero_reduce_scatter_bucket_amp": [vp, vpp, ctypes.c_int, ctypes.c_int, vpp, hp,
                                                   vp, vp, i64, u64, i64, i64, vp],
                "zero_step_amp_noalloc": [vp, vpp, ctypes.c_int, ctypes.c_int, vpp, vpp, vpp,
                                          vpp, vp, vpp, hp, ctypes.POINTER(AmpConfigC), vp, u64,
                                          i64, vp],
                "zero_zero3_pass": [vp, ctypes.POINTER(_LayerC), i32, vpp, i32, ctypes.c_int,
                                    ctypes.c_int, hp, i64, vp, vp],
            }
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.zero_plan_destroy.argtypes = [vp]
            L.zero_plan_destroy.restype = None
            L.zero_last_error.restype = ctypes.c_char_p
            L.zero_version.restype = ctypes.c_char_p
            L.zero_launch_count.restype = i64
            _lib = L
    return _lib


def _check(status: int):
    if status != ZERO_OK:
        raise ZeroError(status, zero_last_error())


def zero_last_error() -> str:
    return lib().zero_last_error().decode()


def zero_version() -> str:
    return lib().zero_version().decode()


def zero_launch_count() -> int:
    return int(lib().zero_launch_count())


# ----------------------------------------------------------------------------
# plan


class Plan:
    """Owner of a zero_plan* (released when garbage-collected)."""

    def __init__(self, handle: int, numel):
        self._h = ctypes.c_void_p(handle)
        self.numel = tuple(int(x) for x in numel)
        n, mode, align, nt = (ctypes.c_int32() for _ in range(4))
        _check(lib().zero_plan_info(self._h, ctypes.byref(n), ctypes.byref(mode),
                                    ctypes.byref(align), ctypes.byref(nt)))
        self.n_ranks, self.mode, self.align = n.value, mode.value, align.value
        phi, padded = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().zero_plan_total(self._h, ctypes.byref(phi), ctypes.byref(padded)))
        self.phi, self.padded = phi.value, padded.value
        self.shards = [self._shard(r) for r in range(self.n_ranks)]
        self._seg_cache = {}

    @property
    def handle(self):
        return self._h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.zero_plan_destroy(h)
            self._h = None

    def _shard(self, r):
        off, ln = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().zero_plan_shard(self._h, r, ctypes.byref(off), ctypes.byref(ln)))
        return off.value, ln.value

    def shard_len(self, r: int) -> int:
        return self.shards[r][1]

    def segments(self, r: int) -> np.ndarray:
        """Rows (tensor_idx, tensor_off, flat_off, shard_off, len) of rank r."""
        if r in self._seg_cache:
            return self._seg_cache[r]
        n = ctypes.c_int64()
        _check(lib().zero_plan_segments(self._h, r, None, None, None, None, None, 0,
                                        ctypes.byref(n)))
        out = np.zeros((5, max(1, n.value)), np.int64)
        ptrs = [out[i].ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) for i in range(5)]
        _check(lib().zero_plan_segments(self._h, r, *ptrs, n.value, ctypes.byref(n)))
        seg = out[:, :n.value].T.copy()
        self._seg_cache[r] = seg
        return seg

    def flat_extent(self, mask: int) -> int:
        """One past the largest flat index owned by a rank in mask."""
        ext = 0
        for r in range(self.n_ranks):
            if (mask >> r) & 1:
                seg = self.segments(r)
                if len(seg):
                    ext = max(ext, int((seg[:, 2] + seg[:, 4]).max()))
        return ext

    def describe(self) -> str:
        buf = ctypes.create_string_buffer(1 << 16)
        _check(lib().zero_plan_describe(self._h, buf, len(buf)))
        return buf.value.decode()

    @property
    def all_ranks(self) -> int:
        return (1 << self.n_ranks) - 1


def zero_plan_partitions(numel: Sequence[int], n_ranks: int, mode="flat",
                         align_elems: int = 16) -> Plan:
    arr = (ctypes.c_int64 * max(1, len(numel)))(*[int(x) for x in numel])
    mode_i = _MODES[mode] if isinstance(mode, str) else int(mode)
    out = ctypes.c_void_p()
    _check(lib().zero_plan_partitions(arr, len(numel), n_ranks, mode_i, align_elems,
                                      ctypes.byref(out)))
    return Plan(out.value, numel)


def zero_memory_bytes(stage: int, phi: int, n_ranks: int):
    num, den = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().zero_memory_bytes(stage, phi, n_ranks, ctypes.byref(num), ctypes.byref(den)))
    return num.value, den.value


# ----------------------------------------------------------------------------
# marshalling


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return ZERO_FP16
    if t.dtype == torch.bfloat16:
        return ZERO_BF16
    raise TypeError(f"expected a float16 or bfloat16 tensor, got {t.dtype}")


def _addr(t, what: str, min_numel: Optional[int] = None, dtype=None) -> int:
    """Device address of a tensor (or pass-through of an int address)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what}: expected a torch.Tensor or an int address")
    if t.numel() == 0 and (min_numel or 0) == 0:
        return 0  # an empty buffer is never touched (and an empty host tensor reports unpinned)
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{what}: tensor must be on a CUDA device or in pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{what}: tensor must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what}: expected {dtype}, got {t.dtype}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{what}: has {t.numel()} elements, needs at least {min_numel}")
    return t.data_ptr()


def _ptrs(values):
    return (ctypes.c_void_p * max(1, len(values)))(*[v or None for v in values])


def _stream(stream) -> Optional[int]:
    if stream is None:
        torch = _torch()
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _mask(plan: Plan, rank_mask) -> int:
    return plan.all_ranks if rank_mask is None else int(rank_mask)


def _per_rank(plan, seq, what, mask, dtype=None, nullable=False, sized=True):
    if seq is None:
        raise ValueError(f"{what}: a list of {plan.n_ranks} entries is required")
    if len(seq) != plan.n_ranks:
        raise ValueError(f"{what}: expected {plan.n_ranks} entries, got {len(seq)}")
    out = []
    for r, t in enumerate(seq):
        if not (mask >> r) & 1:
            out.append(0)
            continue
        if t is None and nullable:
            out.append(0)
            continue
        if t is None:
            raise ValueError(f"{what}[{r}] is None for a masked rank")
        out.append(_addr(t, f"{what}[{r}]", plan.shard_len(r) if sized else None, dtype))
    return out


def _sixteen(seq):
    for t in seq:
        if t is not None and not isinstance(t, int):
            return _dtype_code(t)
    raise ValueError("cannot infer the 16-bit dtype: pass dtype=")


# ----------------------------------------------------------------------------
# device calls


def zero_init_shards(plan: Plan, full_flat16, master, m, v, rank_mask=None, stream=None,
                     dtype=None):
    torch = _torch()
    mask = _mask(plan, rank_mask)
    dt = _dtype_code(full_flat16) if dtype is None else dtype
    full = _addr(full_flat16, "full_flat16", plan.flat_extent(mask))
    ms = _per_rank(plan, master, "master", mask, torch.float32)
    mm = _per_rank(plan, m, "m", mask, torch.float32)
    vv = _per_rank(plan, v, "v", mask, torch.float32)
    _check(lib().zero_init_shards(plan.handle, full, dt, _ptrs(ms), _ptrs(mm), _ptrs(vv), mask,
                                  _stream(stream)))


def zero_reduce_scatter(plan: Plan, grads, op, grad_shards, rank_mask=None, bucket_elems=0,
                        stream=None, dtype=None):
    torch = _torch()
    mask = _mask(plan, rank_mask)
    dt = _sixteen(grads) if dtype is None else dtype
    ext = plan.flat_extent(mask)
    if len(grads) != plan.n_ranks:
        raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
    g = [_addr(t, f"grads[{q}]", ext) for q, t in enumerate(grads)]
    out = _per_rank(plan, grad_shards, "grad_shards", mask, torch.float32)
    op_i = _OPS[op] if isinstance(op, str) else int(op)
    _check(lib().zero_reduce_scatter(plan.handle, _ptrs(g), dt, op_i, _ptrs(out), mask,
                                     int(bucket_elems), _stream(stream)))


def zero_adamw_shard_step(plan: Plan, master, m, v, grad_shards, out16_shard, hparams: AdamW,
                          step: int, rank_mask=None, stream=None, dtype=None):
    torch = _torch()
    mask = _mask(plan, rank_mask)
    ms = _per_rank(plan, master, "master", mask, torch.float32)
    mm = _per_rank(plan, m, "m", mask, torch.float32)
    vv = _per_rank(plan, v, "v", mask, torch.float32)
    gs = _per_rank(plan, grad_shards, "grad_shards", mask, torch.float32)
    if out16_shard is not None:
        dt = _sixteen(out16_shard) if dtype is None else dtype
        o16 = _ptrs(_per_rank(plan, out16_shard, "out16_shard", mask, nullable=True))
    else:
        if dtype is None:
            raise ValueError("dtype is required when out16_shard is None")
        dt, o16 = dtype, None
    hp = hparams.c()
    _check(lib().zero_adamw_shard_step(plan.handle, _ptrs(ms), _ptrs(mm), _ptrs(vv), _ptrs(gs),
                                       o16, dt, ctypes.byref(hp), int(step), mask,
                                       _stream(stream)))


def zero_allgather(plan: Plan, shards16, full_flat16, rank_mask=None, stream=None, dtype=None):
    mask = _mask(plan, rank_mask)
    dt = _dtype_code(full_flat16) if dtype is None else dtype
    sh = _per_rank(plan, shards16, "shards16", mask)
    full = _addr(full_flat16, "full_flat16", plan.flat_extent(mask))
    _check(lib().zero_allgather(plan.handle, _ptrs(sh), dt, full, mask, _stream(stream)))


def zero_step(plan: Plan, grads, op, master, m, v, full_flat16, out16_shard, hparams: AdamW,
              step: int, rank_mask=None, bucket_elems=0, stream=None, dtype=None):
    """The fused reduce-scatter + AdamW + cast + all-gather (see zero.h)."""
    torch = _torch()
    mask = _mask(plan, rank_mask)
    dt = _sixteen(grads) if dtype is None else dtype
    ext = plan.flat_extent(mask)
    if len(grads) != plan.n_ranks:
        raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
    g = [_addr(t, f"grads[{q}]", ext) for q, t in enumerate(grads)]
    ms = _per_rank(plan, master, "master", mask, torch.float32)
    mm = _per_rank(plan, m, "m", mask, torch.float32)
    vv = _per_rank(plan, v, "v", mask, torch.float32)
    full = _addr(full_flat16, "full_flat16", ext) if full_flat16 is not None else None
    o16 = (_ptrs(_per_rank(plan, out16_shard, "out16_shard", mask, nullable=True))
           if out16_shard is not None else None)
    op_i = _OPS[op] if isinstance(op, str) else int(op)
    hp = hparams.c()
    _check(lib().zero_step(plan.handle, _ptrs(g), dt, op_i, _ptrs(ms), _ptrs(mm), _ptrs(vv),
                           full, o16, ctypes.byref(hp), int(step), mask, int(bucket_elems),
                           _stream(stream)))


def zero_floor_probe(plan: Plan, kind: int, grads, master, m, v, full_flat16, rank_mask=None,
                     bucket_elems=0, stream=None, dtype=None):
    """Launches with zero_step's grid and memory accesses but none of its
    arithmetic (kind 0: launch only; 1: loads; 2: loads and stores), for
    timing the floor of a launch of that shape (see zero.h)."""
    torch = _torch()
    mask = _mask(plan, rank_mask)
    dt = _sixteen(grads) if dtype is None else dtype
    ext = plan.flat_extent(mask)
    if len(grads) != plan.n_ranks:
        raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
    g = [_addr(t, f"grads[{q}]", ext) for q, t in enumerate(grads)]
    ms = _per_rank(plan, master, "master", mask, torch.float32)
    mm = _per_rank(plan, m, "m", mask, torch.float32)
    vv = _per_rank(plan, v, "v", mask, torch.float32)
    full = _addr(full_flat16, "full_flat16", ext) if full_flat16 is not None else None
    _check(lib().zero_floor_probe(plan.handle, int(kind), _ptrs(g), dt, _ptrs(ms), _ptrs(mm),
                                  _ptrs(vv), full, mask, int(bucket_elems), _stream(stream)))


def zero_sync(stream=None):
    _check(lib().zero_sync(_stream(stream)))


class ZeroStep:
    """A prepared fused step: the pointer arrays of one set of buffers are
    marshalled once, and each call passes them straight to zero_step.  Used
    where per-call Python overhead would show next to the kernel (benchmark
    loops, the ZeRO-3 layer stream)."""

    def __init__(self, plan: Plan, grads, op, master, m, v, full_flat16, out16_shard,
                 hparams: AdamW, rank_mask=None, bucket_elems=0, dtype=None):
        torch = _torch()
        mask = _mask(plan, rank_mask)
        self.plan, self.mask, self.bucket = plan, mask, int(bucket_elems)
        self.dt = _sixteen(grads) if dtype is None else dtype
        ext = plan.flat_extent(mask)
        if len(grads) != plan.n_ranks:
            raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
        self._g = _ptrs([_addr(t, f"grads[{q}]", ext) for q, t in enumerate(grads)])
        self._ms = _ptrs(_per_rank(plan, master, "master", mask, torch.float32))
        self._mm = _ptrs(_per_rank(plan, m, "m", mask, torch.float32))
        self._vv = _ptrs(_per_rank(plan, v, "v", mask, torch.float32))
        self._full = _addr(full_flat16, "full_flat16", ext) if full_flat16 is not None else None
        self._o16 = (_ptrs(_per_rank(plan, out16_shard, "out16_shard", mask, nullable=True))
                     if out16_shard is not None else None)
        self.op = _OPS[op] if isinstance(op, str) else int(op)
        self._hp = hparams.c()
        self._keep = (grads, master, m, v, full_flat16, out16_shard)

    def __call__(self, step: int, stream=None):
        _check(lib().zero_step(self.plan.handle, self._g, self.dt, self.op, self._ms, self._mm,
                               self._vv, self._full, self._o16, ctypes.byref(self._hp),
                               int(step), self.mask, self.bucket, _stream(stream)))


class FloorProbe:
    """zero_floor_probe with its pointer arrays marshalled once (as ZeroStep),
    so that timing loops measure the launches, not the marshalling."""

    def __init__(self, plan: Plan, kind: int, grads, master, m, v, full_flat16, rank_mask=None,
                 bucket_elems=0, dtype=None):
        torch = _torch()
        mask = _mask(plan, rank_mask)
        self.plan, self.kind, self.mask, self.bucket = plan, int(kind), mask, int(bucket_elems)
        self.dt = _sixteen(grads) if dtype is None else dtype
        ext = plan.flat_extent(mask)
        if len(grads) != plan.n_ranks:
            raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
        self._g = _ptrs([_addr(t, f"grads[{q}]", ext) for q, t in enumerate(grads)])
        self._ms = _ptrs(_per_rank(plan, master, "master", mask, torch.float32))
        self._mm = _ptrs(_per_rank(plan, m, "m", mask, torch.float32))
        self._vv = _ptrs(_per_rank(plan, v, "v", mask, torch.float32))
        self._full = _addr(full_flat16, "full_flat16", ext) if full_flat16 is not None else None
        self._keep = (grads, master, m, v, full_flat16)

    def __call__(self, stream=None):
        _check(lib().zero_floor_probe(self.plan.handle, self.kind, self._g, self.dt, self._ms,
                                      self._mm, self._vv, self._full, self.mask, self.bucket,
                                      _stream(stream)))


# ----------------------------------------------------------------------------
# mixed-precision controls


class AmpConfigC(ctypes.Structure):
    _fields_ = [("init_scale", ctypes.c_double), ("min_scale", ctypes.c_double),
                ("window", ctypes.c_int32), ("hysteresis", ctypes.c_int32),
                ("max_norm", ctypes.c_double)]


class AmpState(ctypes.Structure):
    """Host image of zero_amp_state (80 bytes)."""
    _fields_ = [("scale", ctypes.c_double), ("norm", ctypes.c_double),
                ("step", ctypes.c_int64), ("skipped", ctypes.c_int64),
                ("good_steps", ctypes.c_int32), ("hysteresis_left", ctypes.c_int32),
                ("overflow", ctypes.c_int32), ("coef", ctypes.c_float),
                ("sc", ctypes.c_float * 8)]


AMP_STATE_BYTES = ctypes.sizeof(AmpState)


@dataclasses.dataclass
class AmpConfig:
    init_scale: float = 65536.0
    min_scale: float = 1.0
    window: int = 1000
    hysteresis: int = 2
    max_norm: float = 0.0

    def c(self) -> AmpConfigC:
        return AmpConfigC(self.init_scale, self.min_scale, self.window, self.hysteresis,
                          self.max_norm)


def amp_state_tensor(device="cuda"):
    """Device buffer for a zero_amp_state (torch allocations are 256-byte aligned)."""
    torch = _torch()
    return torch.zeros(AMP_STATE_BYTES, dtype=torch.uint8, device=device)


def read_amp_state(d_state) -> AmpState:
    """Copy the device state to the host (synchronizes with the current stream)."""
    raw = d_state.detach().cpu().numpy().tobytes()
    return AmpState.from_buffer_copy(raw)


def zero_amp_init(d_state, cfg: AmpConfig, stream=None):
    L = lib()
    L.zero_amp_init.argtypes = [ctypes.c_void_p, ctypes.POINTER(AmpConfigC), ctypes.c_void_p]
    L.zero_amp_init.restype = ctypes.c_int
    c = cfg.c()
    _check(L.zero_amp_init(_addr(d_state, "d_state", AMP_STATE_BYTES), ctypes.byref(c),
                           _stream(stream)))


def zero_amp_workspace_bytes(plan: Plan, rank_mask=None, bucket_elems=0) -> int:
    L = lib()
    L.zero_amp_workspace_bytes.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int64,
                                           ctypes.POINTER(ctypes.c_int64)]
    L.zero_amp_workspace_bytes.restype = ctypes.c_int
    out = ctypes.c_int64()
    _check(L.zero_amp_workspace_bytes(plan.handle, _mask(plan, rank_mask), int(bucket_elems),
                                      ctypes.byref(out)))
    return out.value


def zero_step_amp(plan: Plan, grads, op, grad_shards, master, m, v, full_flat16, out16_shard,
                  hparams: AdamW, cfg: AmpConfig, d_state, workspace, rank_mask=None,
                  bucket_elems=0, stream=None, dtype=None):
    """Mixed-precision step: loss-scale check, clipping, AdamW, cast, gather."""
    torch = _torch()
    L = lib()
    vp, vpp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
    L.zero_step_amp.argtypes = [vp, vpp, ctypes.c_int, ctypes.c_int, vpp, vpp, vpp, vpp, vp, vpp,
                                ctypes.POINTER(AdamWHparams), ctypes.POINTER(AmpConfigC), vp, vp,
                                ctypes.c_int64, ctypes.c_uint64, ctypes.c_int64, vp]
    L.zero_step_amp.restype = ctypes.c_int
    mask = _mask(plan, rank_mask)
    dt = _sixteen(grads) if dtype is None else dtype
    ext = plan.flat_extent(mask)
    if len(grads) != plan.n_ranks:
        raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
    g = [_addr(t, f"grads[{q}]", ext) for q, t in enumerate(grads)]
    gs = _per_rank(plan, grad_shards, "grad_shards", mask, torch.float32)
    ms = _per_rank(plan, master, "master", mask, torch.float32)
    mm = _per_rank(plan, m, "m", mask, torch.float32)
    vv = _per_rank(plan, v, "v", mask, torch.float32)
    full = _addr(full_flat16, "full_flat16", ext) if full_flat16 is not None else None
    o16 = (_ptrs(_per_rank(plan, out16_shard, "out16_shard", mask, nullable=True))
           if out16_shard is not None else None)
    need = zero_amp_workspace_bytes(plan, mask, bucket_elems)
    ws_bytes = workspace.numel() * workspace.element_size() if not isinstance(workspace, int) \
        else need
    ws = _addr(workspace, "workspace")
    op_i = _OPS[op] if isinstance(op, str) else int(op)
    hp = hparams.c()
    c = cfg.c()
    _check(L.zero_step_amp(plan.handle, _ptrs(g), dt, op_i, _ptrs(gs), _ptrs(ms), _ptrs(mm),
                           _ptrs(vv), full, o16, ctypes.byref(hp), ctypes.byref(c),
                           _addr(d_state, "d_state", AMP_STATE_BYTES), ws, ws_bytes, mask,
                           int(bucket_elems), _stream(stream)))


def zero_step_amp_shards(plan: Plan, grad_shards, master, m, v, full_flat16, out16_shard,
                         hparams: AdamW, cfg: AmpConfig, d_state, workspace, rank_mask=None,
                         bucket_elems=0, stream=None, dtype=None, _entry="zero_step_amp_shards"):
    """The mixed-precision step from already reduce-scattered fp32 gradient
    shards (read only): loss-scale check, clipping, AdamW, cast, gather.
    ``dtype`` (the 16-bit format) defaults to that of ``full_flat16`` or of
    the first ``out16_shard`` tensor."""
    torch = _torch()
    L = lib()
    mask = _mask(plan, rank_mask)
    ext = plan.flat_extent(mask)
    if dtype is None:
        seq = [full_flat16] + (list(out16_shard) if out16_shard is not None else [])
        dt = _sixteen([t for t in seq if t is not None] or [None])
    else:
        dt = dtype
    gs = _per_rank(plan, grad_shards, "grad_shards", mask, torch.float32)
    ms = _per_rank(plan, master, "master", mask, torch.float32)
    mm = _per_rank(plan, m, "m", mask, torch.float32)
    vv = _per_rank(plan, v, "v", mask, torch.float32)
    full = _addr(full_flat16, "full_flat16", ext) if full_flat16 is not None else None
    o16 = (_ptrs(_per_rank(plan, out16_shard, "out16_shard", mask, nullable=True))
           if out16_shard is not None else None)
    need = zero_amp_workspace_bytes(plan, mask, bucket_elems)
    ws_bytes = workspace.numel() * workspace.element_size() if not isinstance(workspace, int) \
        else need
    ws = _addr(workspace, "workspace")
    hp = hparams.c()
    c = cfg.c()
    _check(getattr(L, _entry)(plan.handle, dt, _ptrs(gs), _ptrs(ms), _ptrs(mm), _ptrs(vv),
                              full, o16, ctypes.byref(hp), ctypes.byref(c),
                              _addr(d_state, "d_state", AMP_STATE_BYTES), ws, ws_bytes, mask,
                              int(bucket_elems), _stream(stream)))


def zero_step_amp_reduced(plan: Plan, grad_shards, master, m, v, full_flat16, out16_shard,
                          hparams: AdamW, cfg: AmpConfig, d_state, workspace, rank_mask=None,
                          bucket_elems=0, stream=None, dtype=None):
    """The mixed-precision step after every bucket was reduced by
    zero_reduce_scatter_bucket_amp (same mask and bucket size): decision and
    update only (see zero.h)."""
    zero_step_amp_shards(plan, grad_shards, master, m, v, full_flat16, out16_shard, hparams, cfg,
                         d_state, workspace, rank_mask, bucket_elems, stream, dtype,
                         _entry="zero_step_amp_reduced")


class ReduceScatterBucketAmp:
    """zero_reduce_scatter_bucket_amp with its pointer arrays marshalled once:
    call(bucket_index, stream) reduces one bucket into the fp32 shards and
    writes its per-tile sums of squares into the workspace."""

    def __init__(self, plan: Plan, grads, op, grad_shards, hparams: AdamW, d_state, workspace,
                 rank_mask=None, bucket_elems=0, dtype=None):
        torch = _torch()
        mask = _mask(plan, rank_mask)
        self.plan, self.mask, self.bucket = plan, mask, int(bucket_elems)
        self.dt = _sixteen(grads) if dtype is None else dtype
        ext = plan.flat_extent(mask)
        if len(grads) != plan.n_ranks:
            raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
        self._g = _ptrs([_addr(t, f"grads[{q}]", ext) for q, t in enumerate(grads)])
        self._gs = _ptrs(_per_rank(plan, grad_shards, "grad_shards", mask, torch.float32))
        self.op = _OPS[op] if isinstance(op, str) else int(op)
        self._hp = hparams.c()
        self._state = _addr(d_state, "d_state", AMP_STATE_BYTES)
        need = zero_amp_workspace_bytes(plan, mask, bucket_elems)
        self._ws_bytes = (workspace.numel() * workspace.element_size()
                          if not isinstance(workspace, int) else need)
        self._ws = _addr(workspace, "workspace")
        self._keep = (grads, grad_shards, d_state, workspace)

    def __call__(self, bucket_index: int, stream=None):
        _check(lib().zero_reduce_scatter_bucket_amp(
            self.plan.handle, self._g, self.dt, self.op, self._gs, ctypes.byref(self._hp),
            self._state, self._ws, self._ws_bytes, self.mask, self.bucket, int(bucket_index),
            _stream(stream)))


def zero_reduce_scatter_bucket_amp(plan: Plan, grads, op, grad_shards, hparams: AdamW, d_state,
                                   workspace, bucket_index: int, rank_mask=None, bucket_elems=0,
                                   stream=None, dtype=None):
    """One bucket of the reduce-scatter that also writes its tiles' sums of
    squares for zero_step_amp_reduced (see zero.h)."""
    ReduceScatterBucketAmp(plan, grads, op, grad_shards, hparams, d_state, workspace,
                           rank_mask, bucket_elems, dtype)(bucket_index, stream)


def zero_step_amp_noalloc(plan: Plan, grads, op, grad_shards, master, m, v, full_flat16,
                          out16_shard, hparams: AdamW, cfg: AmpConfig, d_state, rank_mask=None,
                          bucket_elems=0, stream=None, dtype=None):
    """zero_step_amp for callers that cannot allocate device memory: the
    scratch is the library's fixed 2 MiB device array (steps of up to
    130,560 tiles of 2048 elements).  The first call on a device sets the
    array up (make it before any stream capture); calls that overlap on the
    GPU share the array and must be serialised by the caller."""
    torch = _torch()
    L = lib()
    vp, vpp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
    L.zero_step_amp_noalloc.argtypes = [vp, vpp, ctypes.c_int, ctypes.c_int, vpp, vpp, vpp, vpp,
                                        vp, vpp, ctypes.POINTER(AdamWHparams),
                                        ctypes.POINTER(AmpConfigC), vp, ctypes.c_uint64,
                                        ctypes.c_int64, vp]
    L.zero_step_amp_noalloc.restype = ctypes.c_int
    mask = _mask(plan, rank_mask)
    dt = _sixteen(grads) if dtype is None else dtype
    ext = plan.flat_extent(mask)
    if len(grads) != plan.n_ranks:
        raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
    g = [_addr(t, f"grads[{q}]", ext) for q, t in enumerate(grads)]
    gs = _per_rank(plan, grad_shards, "grad_shards", mask, torch.float32)
    ms = _per_rank(plan, master, "master", mask, torch.float32)
    mm = _per_rank(plan, m, "m", mask, torch.float32)
    vv = _per_rank(plan, v, "v", mask, torch.float32)
    full = _addr(full_flat16, "full_flat16", ext) if full_flat16 is not None else None
    o16 = (_ptrs(_per_rank(plan, out16_shard, "out16_shard", mask, nullable=True))
           if out16_shard is not None else None)
    op_i = _OPS[op] if isinstance(op, str) else int(op)
    hp = hparams.c()
    c = cfg.c()
    _check(L.zero_step_amp_noalloc(plan.handle, _ptrs(g), dt, op_i, _ptrs(gs), _ptrs(ms),
                                   _ptrs(mm), _ptrs(vv), full, o16, ctypes.byref(hp),
                                   ctypes.byref(c), _addr(d_state, "d_state", AMP_STATE_BYTES),
                                   mask, int(bucket_elems), _stream(stream)))


# ----------------------------------------------------------------------------
# ZeRO-3 layer stream


class _LayerC(ctypes.Structure):
    _fields_ = [("grads", ctypes.POINTER(ctypes.c_void_p)),
                ("master", ctypes.POINTER(ctypes.c_void_p)),
                ("m", ctypes.POINTER(ctypes.c_void_p)),
                ("v", ctypes.POINTER(ctypes.c_void_p)),
                ("shards16", ctypes.POINTER(ctypes.c_void_p))]


class Zero3Pass:
    """A prepared ZeRO-3 pass over a stack of layers sharing one plan.

    layers: sequence of dicts with keys grads, master, m, v, shards16 (each a
    list of n_ranks tensors); layer_bufs: the 16-bit layer buffers the gathers
    write, used round-robin (two or more let gathers run ahead)."""

    def __init__(self, plan: Plan, layers, layer_bufs, op, hparams: AdamW, dtype=None):
        torch = _torch()
        all_mask = plan.all_ranks
        self.plan = plan
        self._arrays = []
        self._layers = (_LayerC * len(layers))()
        dt = None
        for i, L in enumerate(layers):
            if len(L["grads"]) != plan.n_ranks:
                raise ValueError(f"layer {i}: expected {plan.n_ranks} gradient replicas")
            g = _ptrs([_addr(t, f"layer {i} grads[{q}]", plan.padded)
                       for q, t in enumerate(L["grads"])])
            parts = [g]
            for key in ("master", "m", "v"):
                parts.append(_ptrs(_per_rank(plan, L[key], f"layer {i} {key}", all_mask,
                                             torch.float32)))
            parts.append(_ptrs(_per_rank(plan, L["shards16"], f"layer {i} shards16", all_mask)))
            self._arrays.append(parts)
            vpp = ctypes.POINTER(ctypes.c_void_p)
            self._layers[i] = _LayerC(*[ctypes.cast(a, vpp) for a in parts])
            if dt is None:
                dt = _sixteen(L["grads"]) if dtype is None else dtype
        self.dt = dt
        self._bufs = _ptrs([_addr(b, f"layer_bufs[{k}]", plan.padded)
                            for k, b in enumerate(layer_bufs)])
        self.n_layers, self.n_bufs = len(layers), len(layer_bufs)
        self.op = _OPS[op] if isinstance(op, str) else int(op)
        self._hp = hparams.c()
        self._keep = (layers, layer_bufs)
        L_ = lib()
        L_.zero_zero3_pass.argtypes = [ctypes.c_void_p, ctypes.POINTER(_LayerC), ctypes.c_int32,
                                       ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32,
                                       ctypes.c_int, ctypes.c_int, ctypes.POINTER(AdamWHparams),
                                       ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        L_.zero_zero3_pass.restype = ctypes.c_int

    def __call__(self, step: int, gather_stream=None, step_stream=None):
        ss = _stream(step_stream)
        gs = _stream(gather_stream) if gather_stream is not None else ss
        _check(lib().zero_zero3_pass(self.plan.handle, self._layers, self.n_layers, self._bufs,
                                     self.n_bufs, self.dt, self.op, ctypes.byref(self._hp),
                                     int(step), gs, ss))


def zero_zero3_pass(plan: Plan, layers, layer_bufs, op, hparams: AdamW, step: int,
                    gather_stream=None, step_stream=None, dtype=None):
    """One ZeRO-3 pass (see include/zero.h); one-shot form of Zero3Pass."""
    Zero3Pass(plan, layers, layer_bufs, op, hparams, dtype)(step, gather_stream, step_stream)


def zero_reduce_scatter_range(plan: Plan, grads, op, grad_shards, flat_lo: int, flat_hi: int,
                              rank_mask=None, stream=None, dtype=None):
    """Reduce-scatter of the flat range [flat_lo, flat_hi) only (one bucket)."""
    torch = _torch()
    L = lib()
    vp, vpp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
    L.zero_reduce_scatter_range.argtypes = [vp, vpp, ctypes.c_int, ctypes.c_int, vpp,
                                            ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, vp]
    L.zero_reduce_scatter_range.restype = ctypes.c_int
    mask = _mask(plan, rank_mask)
    dt = _sixteen(grads) if dtype is None else dtype
    if len(grads) != plan.n_ranks:
        raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
    g = [_addr(t, f"grads[{q}]", plan.flat_extent(mask)) for q, t in enumerate(grads)]
    out = _per_rank(plan, grad_shards, "grad_shards", mask, torch.float32)
    op_i = _OPS[op] if isinstance(op, str) else int(op)
    _check(L.zero_reduce_scatter_range(plan.handle, _ptrs(g), dt, op_i, _ptrs(out), mask,
                                       int(flat_lo), int(flat_hi), _stream(stream)))


class ReduceScatterRange:
    """A prepared zero_reduce_scatter_range: the pointer arrays of one set of
    replicas and shards are marshalled once; each call passes a flat range
    (a bucket) and a stream."""

    def __init__(self, plan: Plan, grads, op, grad_shards, rank_mask=None, dtype=None):
        torch = _torch()
        L = lib()
        vp, vpp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
        L.zero_reduce_scatter_range.argtypes = [vp, vpp, ctypes.c_int, ctypes.c_int, vpp,
                                                ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                                vp]
        L.zero_reduce_scatter_range.restype = ctypes.c_int
        self.plan = plan
        self.mask = _mask(plan, rank_mask)
        self.dt = _sixteen(grads) if dtype is None else dtype
        if len(grads) != plan.n_ranks:
            raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
        ext = plan.flat_extent(self.mask)
        self._g = _ptrs([_addr(t, f"grads[{q}]", ext) for q, t in enumerate(grads)])
        self._out = _ptrs(_per_rank(plan, grad_shards, "grad_shards", self.mask, torch.float32))
        self.op = _OPS[op] if isinstance(op, str) else int(op)
        self._keep = (grads, grad_shards)

    def __call__(self, flat_lo: int, flat_hi: int, stream=None):
        _check(lib().zero_reduce_scatter_range(self.plan.handle, self._g, self.dt, self.op,
                                               self._out, self.mask, int(flat_lo), int(flat_hi),
                                               _stream(stream)))


def _host_addr(a, what):
    """Address of a host array (numpy, CPU tensor) or an int."""
    if a is None:
        return 0
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError(f"{what}: array must be contiguous")
        return a.ctypes.data
    torch = _torch()
    if isinstance(a, torch.Tensor):
        if a.is_cuda or not a.is_contiguous():
            raise ValueError(f"{what}: expected a contiguous host tensor")
        return a.data_ptr()
    raise TypeError(f"{what}: expected a numpy array, a host tensor or an int address")


def _host_per_rank(plan: Plan, seq, what: str, mask: int, nullable: bool = False):
    """Pointer array of per-rank host arrays (entries of unmasked ranks, and
    None entries when nullable, become NULL); None -> NULL array."""
    if seq is None:
        return None
    if len(seq) != plan.n_ranks:
        raise ValueError(f"{what}: expected {plan.n_ranks} entries")
    vals = []
    for r, a in enumerate(seq):
        if not (mask >> r) & 1 or (a is None and nullable):
            vals.append(0)
            continue
        n = a.size if isinstance(a, np.ndarray) else (a.numel() if hasattr(a, "numel") else None)
        if n is not None and n < plan.shard_len(r):
            raise ValueError(f"{what}[{r}]: {n} elements, needs {plan.shard_len(r)}")
        vals.append(_host_addr(a, f"{what}[{r}]"))
    return _ptrs(vals)


def zero_cpu_adamw_shard_step(plan: Plan, master, m, v, grad_shards, out16_shard, hparams: AdamW,
                              step: int, dtype: int, rank_mask=None, n_threads: int = 0):
    """ZeRO-Offload's CPU optimizer: AdamW + cast by host threads on host
    buffers (lists of n_ranks host arrays; entries of unmasked ranks ignored)."""
    mask = _mask(plan, rank_mask)

    def arr(seq, what, nullable=False):
        return _host_per_rank(plan, seq, what, mask, nullable)
    hp = hparams.c()
    o16 = arr(out16_shard, "out16_shard", nullable=True)
    _check(lib().zero_cpu_adamw_shard_step(plan.handle, arr(master, "master"), arr(m, "m"),
                                           arr(v, "v"), arr(grad_shards, "grad_shards"), o16,
                                           int(dtype), ctypes.byref(hp), int(step), mask,
                                           int(n_threads)))


def zero_offload_step(plan: Plan, grads, op, grad_shards, master, m, v, out16_shard,
                      full_flat16, hparams: AdamW, step: int, rank_mask=None,
                      chunk_elems: Optional[int] = None, n_threads: int = 0, stream=None,
                      dtype=None):
    """ZeRO-Offload with the CPU optimizer, pipelined over chunks of the flat
    buffer (see zero.h): device reduce-scatter into the pinned host
    grad_shards, host AdamW + cast on the host master/m/v into the pinned
    host out16_shard, device all-gather into full_flat16 (device, or None).
    grads None: grad_shards already hold the reduced gradients.
    chunk_elems None: the flat buffer in 8 chunks; 0: one chunk."""
    torch = _torch()
    mask = _mask(plan, rank_mask)
    dt = _sixteen(grads if grads is not None else out16_shard) if dtype is None else dtype
    ext = plan.flat_extent(mask)
    g = None
    if grads is not None:
        if len(grads) != plan.n_ranks:
            raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
        g = _ptrs([_addr(t, f"grads[{q}]", ext) for q, t in enumerate(grads)])
    gs = _per_rank(plan, grad_shards, "grad_shards", mask, torch.float32)
    o16 = _per_rank(plan, out16_shard, "out16_shard", mask)
    full = _addr(full_flat16, "full_flat16", ext) if full_flat16 is not None else None
    if chunk_elems is None:
        chunk_elems = max(1, -(-plan.padded // 8))
    op_i = _OPS[op] if isinstance(op, str) else int(op)
    hp = hparams.c()
    _check(lib().zero_offload_step(plan.handle, g, dt, op_i, _ptrs(gs),
                                   _host_per_rank(plan, master, "master", mask),
                                   _host_per_rank(plan, m, "m", mask),
                                   _host_per_rank(plan, v, "v", mask),
                                   _ptrs(o16), full, ctypes.byref(hp), int(step), mask,
                                   int(chunk_elems), int(n_threads), _stream(stream)))


def zero_offload_step_amp(plan: Plan, grads, op, grad_shards, master, m, v, out16_shard,
                          full_flat16, hparams: AdamW, cfg: AmpConfig, state, workspace,
                          rank_mask=None, bucket_elems=0, chunk_elems: Optional[int] = None,
                          n_threads: int = 0, stream=None, dtype=None):
    """The mixed-precision step with the optimizer on the host (see zero.h):
    device reduction and decision, host AdamW + cast of the host state into
    the pinned host out16_shard, device gather of each finished chunk.
    grads None: grad_shards and the workspace's sums of squares were written
    by zero_reduce_scatter_bucket_amp with the same bucket_elems."""
    torch = _torch()
    mask = _mask(plan, rank_mask)
    dt = _sixteen(grads if grads is not None else out16_shard) if dtype is None else dtype
    ext = plan.flat_extent(mask)
    g = None
    if grads is not None:
        if len(grads) != plan.n_ranks:
            raise ValueError(f"grads: expected {plan.n_ranks} replicas, got {len(grads)}")
        g = _ptrs([_addr(t, f"grads[{q}]", ext) for q, t in enumerate(grads)])
    gs = _per_rank(plan, grad_shards, "grad_shards", mask, torch.float32)
    o16 = _per_rank(plan, out16_shard, "out16_shard", mask)
    full = _addr(full_flat16, "full_flat16", ext) if full_flat16 is not None else None
    if chunk_elems is None:
        chunk_elems = max(1, -(-plan.padded // 8))
    op_i = _OPS[op] if isinstance(op, str) else int(op)
    hp, c = hparams.c(), cfg.c()
    ws_bytes = workspace.numel() * workspace.element_size() if not isinstance(workspace, int) \
        else zero_amp_workspace_bytes(plan, mask, bucket_elems)
    _check(lib().zero_offload_step_amp(plan.handle, g, dt, op_i, _ptrs(gs),
                                       _host_per_rank(plan, master, "master", mask),
                                       _host_per_rank(plan, m, "m", mask),
                                       _host_per_rank(plan, v, "v", mask),
                                       _ptrs(o16), full, ctypes.byref(hp), ctypes.byref(c),
                                       _addr(state, "d_state", AMP_STATE_BYTES),
                                       _addr(workspace, "workspace"), ws_bytes, mask,
                                       int(bucket_elems), int(chunk_elems), int(n_threads),
                                       _stream(stream)))

# ----------------------------------------------------------------------------
# the plan queries under their C names (the Plan object caches the same data)


def zero_plan_total(plan: Plan):
    """(phi, padded)."""
    return plan.phi, plan.padded


def zero_plan_info(plan: Plan):
    """(n_ranks, mode, align_elems, n_tensors)."""
    return plan.n_ranks, plan.mode, plan.align, len(plan.numel)


def zero_plan_shard(plan: Plan, rank: int):
    """(flat_off, len) of rank `rank`'s shard (flat_off -1 in round-robin mode)."""
    return plan._shard(rank)


def zero_plan_segments(plan: Plan, rank: int) -> np.ndarray:
    """Rows (tensor_idx, tensor_off, flat_off, shard_off, len)."""
    return plan.segments(rank)


def zero_plan_describe(plan: Plan) -> str:
    return plan.describe()


def zero_plan_destroy(plan: Plan):
    """Release the plan now (it is otherwise released when collected)."""
    h = plan._h
    if h is not None and h.value:
        lib().zero_plan_destroy(h)
    plan._h = None


def zero_selftest_wait_timeout(limit_ns: int, stream=None):
    """Launch the timeout self-test kernel; the next zero_sync raises
    ZeroError with status ZERO_ERR_TIMEOUT (see include/zero.h)."""
    L = lib()
    L.zero_selftest_wait_timeout.argtypes = [ctypes.c_int64, ctypes.c_void_p]
    L.zero_selftest_wait_timeout.restype = ctypes.c_int
    _check(L.zero_selftest_wait_timeout(int(limit_ns), _stream(stream)))
