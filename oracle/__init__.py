"""CPU oracle for split-KV attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never does: the two share
no code. The arithmetic lives in ``oracle.c`` (plain C, double precision, one
function per step of the method); this module compiles it with gcc on first use
and marshals numpy / torch arrays into it.

Functions (all host-side, all double precision):
  split_counts(prob)                    -> int32 [total_q]
  split_range(prob, b, q, s)            -> (k_begin, k_end)
  split_ranges(prob)                    -> k_begin, k_end int32 [total_q, S]
  attention(prob, q, k, v, rows=None)   -> out [n, H, d_v], lse [n, H]
  partials(prob, q, k, v, rows=None)    -> o_part [n, H, S, d_v], l_part [n, H, S]
  merge(o_part, l_part, counts)         -> out [n, H, d_v], lse [n, H]
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "oracle.h")]
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, F16, F32, F64 = 0, 1, 2, 3
MASK_NONE, MASK_CAUSAL, MASK_PREFIX_CAUSAL = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared object beside it (plain gcc, no GPU)."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    stale = force or not os.path.exists(_SO) or any(
        os.path.getmtime(s) > os.path.getmtime(_SO) for s in _SRC)
    if stale:
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread",
                        _SRC[0], "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


class _Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("d_qk", ctypes.c_int),
                ("d_v", ctypes.c_int), ("cu_q", ctypes.POINTER(ctypes.c_int32)),
                ("cu_k", ctypes.POINTER(ctypes.c_int32)), ("mask", ctypes.c_int),
                ("prefix_offset", ctypes.c_int), ("last_valid_kv_index", ctypes.c_int),
                ("n_per_block", ctypes.c_int), ("split_kv", ctypes.c_int),
                ("block_m", ctypes.c_int), ("scale", ctypes.c_double),
                ("window_left", ctypes.c_int), ("seqused_k", ctypes.POINTER(ctypes.c_int32))]


class _Array(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int)]


def use_library(path: str | None):
    """Point the wrappers at another build of oracle.c (None: the default build).

    Used by the tests that plant a mistake in a copy of oracle.c and check that
    the pins catch it. Returns the previously loaded handle."""
    global _lib
    with _lock:
        old, _lib = _lib, None
    if path is not None:
        _load(path)
    return old


def _load(path: str | None = None):
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(path or build())
            P, A = ctypes.POINTER(_Problem), _Array
            i32p, f64p = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            lib.orc_check_problem.argtypes = [P]
            lib.orc_last_valid.argtypes = [P, ctypes.c_int]
            lib.orc_visible.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.orc_split_counts.argtypes = [P, i32p]
            lib.orc_split_range.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ip, ip]
            lib.orc_split_ranges.argtypes = [P, i32p, i32p]
            lib.orc_attention.argtypes = [P, A, A, A, i32p, ctypes.c_int, f64p, f64p, ctypes.c_int]
            lib.orc_partials.argtypes = [P, A, A, A, i32p, ctypes.c_int, f64p, f64p, ctypes.c_int]
            lib.orc_merge.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      f64p, f64p, i32p, f64p, f64p]
            _lib = lib
    return _lib


@dataclass
class Problem:
    """Shape and masking of one split-KV attention problem (host-side view).

    cu_q / cu_k are the cumulative sequence lengths ([B+1], starting at 0);
    mask is MASK_NONE / MASK_CAUSAL / MASK_PREFIX_CAUSAL; last_valid_kv_index -1
    means "each sequence's last key"; scale None means 1/sqrt(d_qk); window_left -1 means
    no sliding window; seqused_k (per sequence) shortens padded key slots.
    """
    cu_q: list
    cu_k: list
    H: int
    d_qk: int
    d_v: int
    mask: int = MASK_NONE
    prefix_offset: int = 0
    last_valid_kv_index: int = -1
    n_per_block: int = 128
    split_kv: int = 1
    block_m: int = 256
    scale: float | None = None
    window_left: int = -1
    seqused_k: list | None = None
    _keep: list = field(default_factory=list, repr=False)

    @property
    def B(self) -> int:
        return len(self.cu_q) - 1

    @property
    def total_q(self) -> int:
        return int(self.cu_q[-1])

    @property
    def total_k(self) -> int:
        return int(self.cu_k[-1])

    def c(self) -> _Problem:
        cq = np.ascontiguousarray(np.asarray(self.cu_q, dtype=np.int32))
        ck = np.ascontiguousarray(np.asarray(self.cu_k, dtype=np.int32))
        self._keep = [cq, ck]
        used = None
        if self.seqused_k is not None:
            su = np.ascontiguousarray(np.asarray(self.seqused_k, dtype=np.int32))
            self._keep.append(su)
            used = su.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        scale = self.scale if self.scale is not None else 1.0 / float(np.sqrt(self.d_qk))
        return _Problem(self.B, self.H, self.d_qk, self.d_v,
                        cq.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                        ck.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                        self.mask, self.prefix_offset, self.last_valid_kv_index,
                        self.n_per_block, self.split_kv, self.block_m, scale,
                        self.window_left, used)


def _as_array(x, keep: list) -> _Array:
    """Stored values, as they are (bf16 as raw bits); the C side widens exactly."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                a = x.view(torch.int16).numpy()
                keep.append(a)
                return _Array(a.ctypes.data, BF16)
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    code = {np.dtype(np.float16): F16, np.dtype(np.float32): F32,
            np.dtype(np.float64): F64}.get(a.dtype)
    if code is None:
        raise TypeError(f"oracle: unsupported input dtype {a.dtype}")
    keep.append(a)
    return _Array(a.ctypes.data, code)


def _threads(nthreads):
    return nthreads if nthreads else (os.cpu_count() or 1)


def _rows(prob: Problem, rows):
    if rows is None:
        rows = np.arange(prob.total_q, dtype=np.int32)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int32))


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle: {what} rejected its arguments (rc={rc})")


def last_valid(prob: Problem, b: int) -> int:
    return _load().orc_last_valid(ctypes.byref(prob.c()), b)


def visible(prob: Problem, b: int, q: int, j: int) -> bool:
    return bool(_load().orc_visible(ctypes.byref(prob.c()), b, q, j))


def split_counts(prob: Problem) -> np.ndarray:
    out = np.zeros(prob.total_q, dtype=np.int32)
    _check(_load().orc_split_counts(ctypes.byref(prob.c()),
                                    out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
           "split_counts")
    return out


def split_range(prob: Problem, b: int, q: int, s: int) -> tuple[int, int]:
    kb, ke = ctypes.c_int(), ctypes.c_int()
    _check(_load().orc_split_range(ctypes.byref(prob.c()), b, q, s,
                                   ctypes.byref(kb), ctypes.byref(ke)), "split_range")
    return kb.value, ke.value


def split_ranges(prob: Problem) -> tuple[np.ndarray, np.ndarray]:
    """k_begin, k_end int32 [total_q, S]: split_range for every packed row."""
    kb = np.zeros((prob.total_q, prob.split_kv), dtype=np.int32)
    ke = np.zeros((prob.total_q, prob.split_kv), dtype=np.int32)
    i32p = ctypes.POINTER(ctypes.c_int32)
    _check(_load().orc_split_ranges(ctypes.byref(prob.c()), kb.ctypes.data_as(i32p),
                                    ke.ctypes.data_as(i32p)), "split_ranges")
    return kb, ke


def attention(prob: Problem, q, k, v, rows=None, nthreads=None):
    """Unsplit attention of the listed packed rows: out [n, H, d_v], lse [n, H]."""
    keep: list = []
    r = _rows(prob, rows)
    out = np.zeros((len(r), prob.H, prob.d_v))
    lse = np.zeros((len(r), prob.H))
    f64p = ctypes.POINTER(ctypes.c_double)
    _check(_load().orc_attention(ctypes.byref(prob.c()), _as_array(q, keep), _as_array(k, keep),
                                 _as_array(v, keep),
                                 r.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(r),
                                 out.ctypes.data_as(f64p), lse.ctypes.data_as(f64p),
                                 _threads(nthreads)), "attention")
    return out, lse


def partials(prob: Problem, q, k, v, rows=None, nthreads=None):
    """Split partials of the listed rows: o_part [n, H, S, d_v], l_part [n, H, S]."""
    keep: list = []
    r = _rows(prob, rows)
    S = prob.split_kv
    o = np.zeros((len(r), prob.H, S, prob.d_v))
    lp = np.zeros((len(r), prob.H, S))
    f64p = ctypes.POINTER(ctypes.c_double)
    _check(_load().orc_partials(ctypes.byref(prob.c()), _as_array(q, keep), _as_array(k, keep),
                                _as_array(v, keep),
                                r.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(r),
                                o.ctypes.data_as(f64p), lp.ctypes.data_as(f64p),
                                _threads(nthreads)), "partials")
    return o, lp


def merge(o_part: np.ndarray, l_part: np.ndarray, counts: np.ndarray):
    """NaN-safe merge: o_part [n, H, S, d_v], l_part [n, H, S], counts [n]."""
    o_part = np.ascontiguousarray(o_part, dtype=np.float64)
    l_part = np.ascontiguousarray(l_part, dtype=np.float64)
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    n, H, S, dv = o_part.shape
    out = np.zeros((n, H, dv))
    lse = np.zeros((n, H))
    f64p = ctypes.POINTER(ctypes.c_double)
    _check(_load().orc_merge(n, H, S, dv, o_part.ctypes.data_as(f64p),
                             l_part.ctypes.data_as(f64p),
                             counts.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                             out.ctypes.data_as(f64p), lse.ctypes.data_as(f64p)), "merge")
    return out, lse
