"""CPU oracle of the ZeRO sharded optimizer step -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs anything here, and this
package imports nothing from the product.

The arithmetic lives in ``zero_oracle.c`` (plain single-threaded C, compiled
with ``-ffp-contract=off`` so every binary32 operation rounds once); this
module only compiles it, loads it with ctypes and converts numpy arrays.

Parity status of each function (what pins it; the pins are the ``not gpu``
tests in tests/test_oracle_pins.py):
  plan_flat / segments   brute force on tiny inputs, invariants, the
                         round-robin example of "ZeRO 优化器" (cookllm.com),
                         参数分配策略 (params 0, 4, 8 -> GPU 0)
  memory_bytes           the closed forms of "ZeRO / DeepSpeed 深度解读报告"
                         §3.3 against bytes actually allocated per virtual rank,
                         and the pages' worked numbers (BERT-base 220/880 MB,
                         70B/8 -> 17.5 GB, -87.5 % at N=8, -75 % at N=4)
  f32_to_16 / 16_to_f32  exhaustive over all 2^32 binary32 inputs against
                         numpy (binary16) and torch (bfloat16) conversions
  reduce                 exact sums of scaled small integers; the recursive
                         summation error bound against a binary64 sum
  adamw / update         torch.optim.AdamW at N=1; the first-step closed form;
                         pure decay for zero gradients
  step                   partition invariance (sharded == unsharded, bit for
                         bit) across N, A and both partition modes
  step_amp               S = 1 without clipping == step (bit-exact); a power-of-
                         two loss scale on exactly scaled gradients == step on
                         the unscaled ones (bit-exact); clipping == torch's
                         clip_grad_norm_ followed by torch.optim.AdamW; the
                         loss-scale trajectory of the configuration keys
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FP16, BF16 = 0, 1
FLAT, ROUND_ROBIN = 0, 1
SUM, AVG = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


class Hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("weight_decay", ctypes.c_double)]


def build(force: bool = False) -> str:
    """Compile zero_oracle.c into liboracle.so next to it (host compiler)."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = [os.environ.get("CC", "gcc"), "-O2", "-ffp-contract=off",
               "-fno-fast-math", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            i64p = ctypes.POINTER(ctypes.c_int64)
            L.orc_plan_flat.argtypes = [i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        i64p, i64p, i64p]
            L.orc_segments.argtypes = [i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_int32, i64p, i64p, i64p, i64p,
                                       i64p, ctypes.c_int64, i64p]
            L.orc_memory_bytes.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                           i64p, i64p]
            L.orc_f32_to_16_array.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int64]
            L.orc_16_to_f32_array.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int64]
            L.orc_step_scalars.argtypes = [ctypes.POINTER(Hparams), ctypes.c_int64,
                                           ctypes.c_void_p]
            L.orc_reduce_elements.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
            L.orc_adamw_elements.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.POINTER(Hparams),
                                             ctypes.c_int64]
            L.orc_update_elements.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.POINTER(Hparams), ctypes.c_int64]
            vpp = ctypes.POINTER(ctypes.c_void_p)
            L.orc_step.argtypes = [i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vpp, vpp, vpp,
                                   vpp, ctypes.c_void_p, vpp, ctypes.POINTER(Hparams),
                                   ctypes.c_int64, ctypes.c_uint64]
            L.orc_reduce_scatter.argtypes = [i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vpp,
                                             vpp, ctypes.c_uint64]
            L.orc_allgather.argtypes = [i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, vpp, ctypes.c_void_p, ctypes.c_uint64]
            for name in ("orc_plan_flat", "orc_segments", "orc_memory_bytes", "orc_step",
                         "orc_reduce_scatter", "orc_allgather"):
                getattr(L, name).restype = ctypes.c_int
            for name in ("orc_f32_to_16_array", "orc_16_to_f32_array", "orc_step_scalars",
                         "orc_reduce_elements", "orc_adamw_elements", "orc_update_elements"):
                getattr(L, name).restype = None
            _lib = L
    return _lib


# ----------------------------------------------------------------------------
# helpers


def _i64(a):
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int64))
    return arr, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data


def _ptr_array(arrays):
    vals = [0 if a is None else _ptr(a) for a in arrays]
    return (ctypes.c_void_p * max(1, len(vals)))(*vals)


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01) -> Hparams:
    return Hparams(lr, beta1, beta2, eps, weight_decay)


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"oracle {what} rejected its arguments")


# ----------------------------------------------------------------------------
# plan and memory model


def plan_flat(numel, n_ranks: int, align: int):
    """(phi, P, S) of the near-equal flat partition."""
    arr, p = _i64(numel)
    phi, P, S = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().orc_plan_flat(p, len(arr), n_ranks, align, ctypes.byref(phi),
                               ctypes.byref(P), ctypes.byref(S)), "plan_flat")
    return phi.value, P.value, S.value


def segments(numel, n_ranks: int, mode: int, align: int, rank: int) -> np.ndarray:
    """Rank `rank`'s segments as an int64 array of rows
    (tensor_idx, tensor_off, flat_off, shard_off, len)."""
    arr, p = _i64(numel)
    L = lib()
    cnt = ctypes.c_int64()
    z = np.zeros(1, np.int64)
    zp = z.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    _check(L.orc_segments(p, len(arr), n_ranks, mode, align, rank, zp, zp, zp, zp, zp, 0,
                          ctypes.byref(cnt)), "segments")
    n = cnt.value
    out = np.zeros((5, max(n, 1)), np.int64)
    ptrs = [out[i].ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) for i in range(5)]
    _check(L.orc_segments(p, len(arr), n_ranks, mode, align, rank, *ptrs, n,
                          ctypes.byref(cnt)), "segments")
    return out[:, :n].T.copy()


def shard_len(numel, n_ranks: int, mode: int, align: int, rank: int) -> int:
    seg = segments(numel, n_ranks, mode, align, rank)
    return int(seg[:, 4].sum()) if len(seg) else 0


def flat_len(numel, n_ranks: int, mode: int, align: int) -> int:
    """Length of the gathered flat buffer: P in flat mode, phi in round-robin."""
    if mode == FLAT:
        return plan_flat(numel, n_ranks, align)[1]
    return int(np.sum(np.asarray(numel, dtype=np.int64)))


def memory_bytes(stage: int, phi: int, n_ranks: int):
    """Per-rank model-state bytes as an exact fraction (num, den)."""
    num, den = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().orc_memory_bytes(stage, phi, n_ranks, ctypes.byref(num), ctypes.byref(den)),
           "memory_bytes")
    return num.value, den.value


# ----------------------------------------------------------------------------
# conversions


def f32_to_16(bits_u32: np.ndarray, dtype: int) -> np.ndarray:
    """Round binary32 values (given as uint32 bit patterns) to 16-bit bits."""
    src = np.ascontiguousarray(bits_u32, dtype=np.uint32)
    out = np.empty(src.shape, np.uint16)
    lib().orc_f32_to_16_array(dtype, _ptr(src), _ptr(out), src.size)
    return out


def to_f32(bits_u16: np.ndarray, dtype: int) -> np.ndarray:
    src = np.ascontiguousarray(bits_u16, dtype=np.uint16)
    out = np.empty(src.shape, np.float32)
    lib().orc_16_to_f32_array(dtype, _ptr(src), _ptr(out), src.size)
    return out


def step_scalars(hp: Hparams, t: int) -> np.ndarray:
    """(d, b1, b2, c1, c2, ss, sb, eps) as binary32, for step t."""
    out = np.zeros(8, np.float32)
    lib().orc_step_scalars(ctypes.byref(hp), t, _ptr(out))
    return out


# ----------------------------------------------------------------------------
# element-wise pieces (arrays gathered from anywhere, e.g. sampled indices)


def reduce_elements(grads16: np.ndarray, dtype: int, op: int) -> np.ndarray:
    """grads16: uint16 array of shape (N, n).  Returns binary32 (n,)."""
    g = np.ascontiguousarray(grads16, dtype=np.uint16)
    N, n = g.shape
    out = np.empty(n, np.float32)
    lib().orc_reduce_elements(n, N, dtype, op, _ptr(g), _ptr(out))
    return out


def adamw_elements(g: np.ndarray, master, m, v, dtype: int, hp: Hparams, t: int,
                   out16: np.ndarray | None = None):
    """In place on master/m/v (binary32 contiguous arrays)."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    lib().orc_adamw_elements(g.size, dtype, _ptr(g), _ptr(master), _ptr(m), _ptr(v),
                             0 if out16 is None else _ptr(out16), ctypes.byref(hp), t)


def update_elements(grads16: np.ndarray, master, m, v, dtype: int, op: int, hp: Hparams,
                    t: int, out16: np.ndarray | None = None):
    """Reduce + AdamW + cast on n gathered elements, in place on master/m/v."""
    g = np.ascontiguousarray(grads16, dtype=np.uint16)
    N, n = g.shape
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"] and a.size == n
    lib().orc_update_elements(n, N, dtype, op, _ptr(g), _ptr(master), _ptr(m), _ptr(v),
                              0 if out16 is None else _ptr(out16), ctypes.byref(hp), t)


# ----------------------------------------------------------------------------
# whole-plan operations


def step(numel, n_ranks: int, mode: int, align: int, dtype: int, op: int, grads, master, m, v,
         full16, shard16, hp: Hparams, t: int, rank_mask: int | None = None):
    """One step of every masked rank.  grads: list of N uint16 flat replicas;
    master/m/v: lists of N float32 shard arrays (None for unmasked ranks);
    full16: uint16 flat buffer or None; shard16: list or None."""
    arr, p = _i64(numel)
    if rank_mask is None:
        rank_mask = (1 << n_ranks) - 1
    vpp = ctypes.POINTER(ctypes.c_void_p)
    g = _ptr_array(grads)
    ms, mm, vv = _ptr_array(master), _ptr_array(m), _ptr_array(v)
    sh = _ptr_array(shard16) if shard16 is not None else None
    _check(lib().orc_step(p, len(arr), n_ranks, mode, align, dtype, op,
                          ctypes.cast(g, vpp), ctypes.cast(ms, vpp), ctypes.cast(mm, vpp),
                          ctypes.cast(vv, vpp), 0 if full16 is None else _ptr(full16),
                          None if sh is None else ctypes.cast(sh, vpp), ctypes.byref(hp), t,
                          rank_mask), "step")


def reduce_scatter(numel, n_ranks: int, mode: int, align: int, dtype: int, op: int, grads,
                   out, rank_mask: int | None = None):
    arr, p = _i64(numel)
    if rank_mask is None:
        rank_mask = (1 << n_ranks) - 1
    vpp = ctypes.POINTER(ctypes.c_void_p)
    _check(lib().orc_reduce_scatter(p, len(arr), n_ranks, mode, align, dtype, op,
                                    ctypes.cast(_ptr_array(grads), vpp),
                                    ctypes.cast(_ptr_array(out), vpp), rank_mask),
           "reduce_scatter")


def allgather(numel, n_ranks: int, mode: int, align: int, shard16, full16,
              rank_mask: int | None = None):
    arr, p = _i64(numel)
    if rank_mask is None:
        rank_mask = (1 << n_ranks) - 1
    vpp = ctypes.POINTER(ctypes.c_void_p)
    _check(lib().orc_allgather(p, len(arr), n_ranks, mode, align,
                               ctypes.cast(_ptr_array(shard16), vpp), _ptr(full16), rank_mask),
           "allgather")


# ----------------------------------------------------------------------------
# mixed-precision controls (loss scaling, overflow skip, clipping)


class AmpConfig(ctypes.Structure):
    _fields_ = [("init_scale", ctypes.c_double), ("min_scale", ctypes.c_double),
                ("window", ctypes.c_int32), ("hysteresis", ctypes.c_int32),
                ("max_norm", ctypes.c_double)]


class AmpState(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_double), ("norm", ctypes.c_double),
                ("step", ctypes.c_int64), ("skipped", ctypes.c_int64),
                ("good_steps", ctypes.c_int32), ("hysteresis_left", ctypes.c_int32),
                ("overflow", ctypes.c_int32), ("coef", ctypes.c_float)]


def amp_config(init_scale=65536.0, min_scale=1.0, window=1000, hysteresis=2, max_norm=0.0):
    return AmpConfig(init_scale, min_scale, window, hysteresis, max_norm)


def amp_init(cfg: AmpConfig) -> AmpState:
    L = lib()
    L.orc_amp_init.argtypes = [ctypes.POINTER(AmpConfig), ctypes.POINTER(AmpState)]
    L.orc_amp_init.restype = None
    st = AmpState()
    L.orc_amp_init(ctypes.byref(cfg), ctypes.byref(st))
    return st


def step_amp(numel, n_ranks: int, mode: int, align: int, dtype: int, op: int, grads, master, m,
             v, full16, shard16, hp: Hparams, cfg: AmpConfig, state: AmpState,
             rank_mask: int | None = None):
    """One mixed-precision step (in place on master/m/v/full16 and state)."""
    L = lib()
    vpp = ctypes.POINTER(ctypes.c_void_p)
    i64p = ctypes.POINTER(ctypes.c_int64)
    L.orc_step_amp.argtypes = [i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                               ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vpp, vpp, vpp,
                               vpp, ctypes.c_void_p, vpp, ctypes.POINTER(Hparams),
                               ctypes.POINTER(AmpConfig), ctypes.POINTER(AmpState),
                               ctypes.c_uint64]
    L.orc_step_amp.restype = ctypes.c_int
    arr, p = _i64(numel)
    if rank_mask is None:
        rank_mask = (1 << n_ranks) - 1
    sh = _ptr_array(shard16) if shard16 is not None else None
    _check(L.orc_step_amp(p, len(arr), n_ranks, mode, align, dtype, op,
                          ctypes.cast(_ptr_array(grads), vpp),
                          ctypes.cast(_ptr_array(master), vpp), ctypes.cast(_ptr_array(m), vpp),
                          ctypes.cast(_ptr_array(v), vpp),
                          0 if full16 is None else _ptr(full16),
                          None if sh is None else ctypes.cast(sh, vpp), ctypes.byref(hp),
                          ctypes.byref(cfg), ctypes.byref(state), rank_mask), "step_amp")
