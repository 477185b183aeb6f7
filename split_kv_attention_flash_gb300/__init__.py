"""Split-KV attention forward for NVIDIA GB300 (sm_103a): Python binding.

Thin ctypes marshalling over the C ABI of include/splitkv.h; every step of the
computation runs in the library's CUDA kernels. PyTorch is used only for device
memory and streams. The functions keep the C names:

  sk_valid_split_counts, sk_attn_partial_fwd, sk_combine, sk_attn_fwd,
  sk_attn_fwd_static, sk_attn_fwd_host, sk_host_buffer_bytes, sk_workspace_bytes, sk_auto_split_kv, sk_choose_split_kv,
  sk_default_block_m, sk_partial_kernel_name, sk_status_string, sk_last_cuda_error,
  sk_selftest_bounded_wait, sk_read_device_error

plus `attention(...)`, which allocates the output / workspace with torch and calls
sk_attn_fwd (the one-call entry, with split_kv = 0 meaning automatic).

Tensors: varlen Q/K/V/out are [rows, H, d] (innermost dim contiguous); dense ones
are [B, seq, H, d]. Partial buffers are f32 [H, S, total_q, d_v] and [H, S, total_q];
the final LSE is f32 [H, total_q]; counts are int32 [total_q].
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from dataclasses import dataclass

import torch

from ._build import LIB as _LIB_PATH

MASK_NONE, MASK_CAUSAL, MASK_PREFIX_CAUSAL = 0, 1, 2
SK_BF16, SK_F16, SK_F32 = 0, 1, 2
_DTYPES = {torch.bfloat16: SK_BF16, torch.float16: SK_F16, torch.float32: SK_F32}
_STATUS = {0: "SK_OK", 1: "SK_ERR_INVALID_ARG", 2: "SK_ERR_UNSUPPORTED", 3: "SK_ERR_WORKSPACE",
           4: "SK_ERR_CUDA", 5: "SK_ERR_TIMEOUT"}


class SplitKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == 4:
            code, name = sk_last_cuda_error()
            detail = f"; {name} ({code})"
        super().__init__(f"{where}: {_STATUS.get(status, status)} ({sk_status_string(status)}{detail})")


class _Params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("max_seqlen_q", ctypes.c_int),
                ("max_seqlen_k", ctypes.c_int), ("total_q", ctypes.c_int),
                ("total_k", ctypes.c_int), ("d_qk", ctypes.c_int), ("d_v", ctypes.c_int),
                ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
                ("mask", ctypes.c_int), ("prefix_offset", ctypes.c_int),
                ("last_valid_kv_index", ctypes.c_int), ("n_per_block", ctypes.c_int),
                ("split_kv", ctypes.c_int), ("block_m", ctypes.c_int),
                ("softmax_scale", ctypes.c_float), ("fuse_combine", ctypes.c_int),
                ("window_left", ctypes.c_int), ("seqused_k", ctypes.c_void_p)]


class _Tensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int), ("stride_b", ctypes.c_int64),
                ("stride_row", ctypes.c_int64), ("stride_h", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded CUDA library. There is no fallback: a missing build is an error."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"split-KV CUDA library not built ({_LIB_PATH} missing); run "
                    "split_kv_attention_flash_gb300._build.build() first")
            L = ctypes.CDLL(_LIB_PATH)
            P, T = ctypes.POINTER(_Params), _Tensor
            vp, fp, i32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
            L.sk_valid_split_counts.argtypes = [P, i32p, vp]
            L.sk_attn_partial_fwd.argtypes = [P, T, T, T, fp, fp, vp]
            L.sk_combine.argtypes = [P, fp, fp, i32p, T, fp, vp]
            L.sk_attn_fwd.argtypes = [P, T, T, T, T, fp, vp, ctypes.c_size_t, vp]
            L.sk_workspace_bytes.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
            L.sk_auto_split_kv.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
            L.sk_choose_split_kv.argtypes = [P, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
            L.sk_default_block_m.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
            L.sk_supported_head_dims.argtypes = [ctypes.c_int, ctypes.c_int]
            L.sk_partial_kernel_name.argtypes = [P, T, T, T]
            L.sk_partial_kernel_name.restype = ctypes.c_char_p
            L.sk_status_string.argtypes = [ctypes.c_int]
            L.sk_status_string.restype = ctypes.c_char_p
            L.sk_read_device_error.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.c_int]
            L.sk_last_cuda_error.argtypes = [ctypes.POINTER(ctypes.c_char_p)]
            _lib = L
    return _lib


@dataclass
class Params:
    """Python mirror of sk_params. cu_seqlens_* are device int32 tensors (or raw
    device addresses as ints), or None for the dense layout."""
    B: int
    H: int
    max_seqlen_q: int
    max_seqlen_k: int
    total_q: int
    total_k: int
    d_qk: int
    d_v: int
    cu_seqlens_q: torch.Tensor | None = None
    cu_seqlens_k: torch.Tensor | None = None
    mask: int = MASK_NONE
    prefix_offset: int = 0
    last_valid_kv_index: int = -1
    n_per_block: int = 128
    split_kv: int = 0
    block_m: int = 0
    softmax_scale: float = 0.0
    fuse_combine: int = 0
    window_left: int = -1
    seqused_k: torch.Tensor | None = None

    def c(self) -> _Params:
        def ptr(t):
            if t is None or isinstance(t, int):
                return t
            if t.dtype != torch.int32:
                raise TypeError("cu_seqlens must be int32")
            return t.data_ptr()
        return _Params(self.B, self.H, self.max_seqlen_q, self.max_seqlen_k, self.total_q,
                       self.total_k, self.d_qk, self.d_v, ptr(self.cu_seqlens_q),
                       ptr(self.cu_seqlens_k), self.mask, self.prefix_offset,
                       self.last_valid_kv_index, self.n_per_block, self.split_kv, self.block_m,
                       self.softmax_scale, self.fuse_combine, self.window_left,
                       ptr(self.seqused_k))

    @property
    def dense(self) -> bool:
        return self.cu_seqlens_q is None


def params_for(w, device="cuda", split_kv=None, **overrides) -> Params:
    """Params of a `workloads.Workload` with cu_seqlens on `device`."""
    cu_q = torch.tensor(w.cu_seqlens_q, dtype=torch.int32, device=device)
    cu_k = torch.tensor(w.cu_seqlens_k, dtype=torch.int32, device=device)
    p = Params(B=w.B, H=w.H, max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k,
               total_q=w.total_q, total_k=w.total_k, d_qk=w.d_qk, d_v=w.d_v, cu_seqlens_q=cu_q,
               cu_seqlens_k=cu_k, mask=w.mask, prefix_offset=w.prefix_offset,
               last_valid_kv_index=w.last_valid_kv_index, n_per_block=w.n_per_block,
               split_kv=w.split_kv if split_kv is None else split_kv,
               window_left=w.window_left,
               seqused_k=None if w.seqused_k is None
               else torch.tensor(w.seqused_k, dtype=torch.int32, device=device))
    for k_, v_ in overrides.items():
        setattr(p, k_, v_)
    return p


def tensor_desc(t: torch.Tensor) -> _Tensor:
    """[rows, H, d] (varlen) or [B, seq, H, d] (dense) with a contiguous last dim."""
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() not in (3, 4) or (t.numel() > 0 and t.stride(-1) != 1):
        raise ValueError("expected [rows, H, d] or [B, seq, H, d] with a contiguous last dim")
    if t.dim() == 3:
        sb, sr, sh = 0, t.stride(0), t.stride(1)
    else:
        sb, sr, sh = t.stride(0), t.stride(1), t.stride(2)
    return _Tensor(t.data_ptr(), _DTYPES[t.dtype], sb, sr, sh)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _ok(status: int, where: str):
    if status != 0:
        raise SplitKVError(status, where)


def sk_status_string(status: int) -> str:
    return lib().sk_status_string(status).decode()


def sk_default_block_m(d_qk: int, d_v: int, dtype=SK_BF16) -> int:
    return lib().sk_default_block_m(d_qk, d_v, dtype)


def sk_choose_split_kv(p: Params, sm_count: int) -> int:
    out = ctypes.c_int()
    _ok(lib().sk_choose_split_kv(ctypes.byref(p.c()), sm_count, ctypes.byref(out)),
        "sk_choose_split_kv")
    return out.value


def sk_auto_split_kv(p: Params) -> int:
    out = ctypes.c_int()
    _ok(lib().sk_auto_split_kv(ctypes.byref(p.c()), ctypes.byref(out)), "sk_auto_split_kv")
    return out.value


def sk_workspace_bytes(p: Params) -> int:
    out = ctypes.c_size_t()
    _ok(lib().sk_workspace_bytes(ctypes.byref(p.c()), ctypes.byref(out)), "sk_workspace_bytes")
    return out.value


def sk_partial_kernel_name(p: Params, q, k, v) -> str | None:
    r = lib().sk_partial_kernel_name(ctypes.byref(p.c()), tensor_desc(q), tensor_desc(k),
                                     tensor_desc(v))
    return None if r is None else r.decode()


def sk_valid_split_counts(p: Params, counts: torch.Tensor, stream=None):
    _ok(lib().sk_valid_split_counts(ctypes.byref(p.c()), _ptr(counts), _stream(stream)),
        "sk_valid_split_counts")


def sk_attn_partial_fwd(p: Params, q, k, v, o_part, lse_part, stream=None):
    _ok(lib().sk_attn_partial_fwd(ctypes.byref(p.c()), tensor_desc(q), tensor_desc(k),
                                  tensor_desc(v), _ptr(o_part), _ptr(lse_part), _stream(stream)),
        "sk_attn_partial_fwd")


def sk_combine(p: Params, o_part, lse_part, counts, out, lse_out=None, stream=None):
    _ok(lib().sk_combine(ctypes.byref(p.c()), _ptr(o_part), _ptr(lse_part), _ptr(counts),
                         tensor_desc(out), _ptr(lse_out), _stream(stream)), "sk_combine")


def sk_attn_fwd(p: Params, q, k, v, out, lse_out=None, workspace=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(lib().sk_attn_fwd(ctypes.byref(p.c()), tensor_desc(q), tensor_desc(k), tensor_desc(v),
                          tensor_desc(out), _ptr(lse_out), _ptr(workspace), ws_bytes,
                          _stream(stream)), "sk_attn_fwd")


SK_STATIC_SCRATCH_BYTES = 32 << 20   # mirrors include/splitkv.h


def sk_attn_fwd_static(p: Params, q, k, v, out, lse_out=None, stream=None):
    """sk_attn_fwd without a workspace argument, for callers that cannot allocate:
    the library's own fixed scratch array (SK_STATIC_SCRATCH_BYTES per GPU) holds the
    split partials. Problems that need more scratch raise SK_ERR_WORKSPACE."""
    L = lib()
    fn = L.sk_attn_fwd_static
    fn.argtypes = [ctypes.POINTER(_Params), _Tensor, _Tensor, _Tensor, _Tensor, ctypes.c_void_p,
                   ctypes.c_void_p]
    _ok(fn(ctypes.byref(p.c()), tensor_desc(q), tensor_desc(k), tensor_desc(v), tensor_desc(out),
           _ptr(lse_out), _stream(stream)), "sk_attn_fwd_static")


def sk_host_buffer_bytes(p: Params, dtype: int, with_lse: bool) -> int:
    fn = lib().sk_host_buffer_bytes
    fn.argtypes = [ctypes.POINTER(_Params), ctypes.c_int, ctypes.c_int,
                   ctypes.POINTER(ctypes.c_size_t)]
    out = ctypes.c_size_t()
    _ok(fn(ctypes.byref(p.c()), dtype, int(with_lse), ctypes.byref(out)), "sk_host_buffer_bytes")
    return out.value


def sk_attn_fwd_host(p: Params, q, k, v, out, lse_out=None, device_buffer=None, stream=None):
    """sk_attn_fwd with q, k, v, out (and lse_out) in host memory (contiguous CPU tensors,
    pinned for asynchronous copies); device_buffer is a device uint8 tensor of at least
    sk_host_buffer_bytes() bytes."""
    fn = lib().sk_attn_fwd_host
    fn.argtypes = [ctypes.POINTER(_Params), _Tensor, _Tensor, _Tensor, _Tensor, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    nbytes = 0 if device_buffer is None else device_buffer.numel() * device_buffer.element_size()
    _ok(fn(ctypes.byref(p.c()), tensor_desc(q), tensor_desc(k), tensor_desc(v), tensor_desc(out),
           _ptr(lse_out), _ptr(device_buffer), nbytes, _stream(stream)), "sk_attn_fwd_host")


def sk_last_cuda_error() -> tuple[int, str]:
    name = ctypes.c_char_p()
    code = lib().sk_last_cuda_error(ctypes.byref(name))
    return code, (name.value or b"").decode()


def sk_selftest_bounded_wait(timeout_ns: int, stream=None):
    fn = lib().sk_selftest_bounded_wait
    fn.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]
    _ok(fn(timeout_ns, _stream(stream) if torch.cuda.is_available() else None),
        "sk_selftest_bounded_wait")


def sk_read_device_error(clear: bool = True) -> int:
    code = ctypes.c_int()
    lib().sk_read_device_error(ctypes.byref(code), int(clear))
    return code.value


def attention(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, *,
              mask=MASK_NONE, prefix_offset=0, last_valid_kv_index=-1, n_per_block=128,
              split_kv=0, softmax_scale=0.0, return_lse=False, out=None, stream=None):
    """One-call varlen split-KV attention forward (split_kv 0: automatic).

    Allocates `out` (unless given) and the workspace with torch, then runs
    sk_attn_fwd. Returns out, or (out, lse) with return_lse."""
    p = Params(B=cu_seqlens_q.numel() - 1, H=q.shape[1], max_seqlen_q=max_seqlen_q,
               max_seqlen_k=max_seqlen_k, total_q=q.shape[0], total_k=k.shape[0],
               d_qk=q.shape[2], d_v=v.shape[2], cu_seqlens_q=cu_seqlens_q,
               cu_seqlens_k=cu_seqlens_k, mask=mask, prefix_offset=prefix_offset,
               last_valid_kv_index=last_valid_kv_index, n_per_block=n_per_block,
               split_kv=split_kv, softmax_scale=softmax_scale)
    if out is None:
        out = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=q.dtype, device=q.device)
    lse = (torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=q.device)
           if return_lse else None)
    nbytes = sk_workspace_bytes(p)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device) if nbytes else None
    sk_attn_fwd(p, q, k, v, out, lse, ws, stream)
    return (out, lse) if return_lse else out


def default_scale(d_qk: int) -> float:
    return 1.0 / math.sqrt(d_qk)
