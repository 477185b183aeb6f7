"""sk_attn_fwd_host: the one-call forward with Q, K, V and the output in host memory.

Through the C ABI, against the device entry point (the same kernels on the same inputs:
identical results) and against the f64 oracle at the stated tolerances, with pinned and with
pageable host tensors, with and without an LSE, in the packed and the dense layouts, and two
calls on two streams with two device buffers (the overlapped form a user would run).
"""
from __future__ import annotations

import pytest
import torch

import oracle
import split_kv_attention_flash_gb300 as skv
from split_kv_attention_flash_gb300 import workloads as wl
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DT = {"bf16": skv.SK_BF16, "f16": skv.SK_F16, "f32": skv.SK_F32}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from split_kv_attention_flash_gb300 import _build
    _build.build()
    skv.lib()


CASES = [
    wl.Workload("prefill causal bf16 D192/128", H=3, seqlens_q=(600, 77), seqlens_k=(3000, 500),
                d_qk=192, d_v=128, dtype="bf16", seed=61, n_per_block=128, split_kv=3,
                mask=wl.MASK_CAUSAL),
    wl.Workload("split 1 f16 D128", H=2, seqlens_q=(300,), seqlens_k=(900,), d_qk=128, d_v=128,
                dtype="f16", seed=62, n_per_block=64, split_kv=1),
    wl.Workload("f32 prefix", H=2, seqlens_q=(64, 90), seqlens_k=(256, 300), d_qk=64, d_v=64,
                dtype="f32", seed=63, n_per_block=32, split_kv=4, mask=wl.MASK_PREFIX_CAUSAL,
                prefix_offset=20),
    wl.Workload("decode-like bf16", H=8, seqlens_q=(1,) * 5, seqlens_k=(4000, 17, 0, 900, 64),
                d_qk=128, d_v=128, dtype="bf16", seed=64, n_per_block=128, split_kv=0),
]


def _host_run(w, q, k, v, pinned=True, with_lse=True, stream=None, buf=None, keep=None):
    """Runs sk_attn_fwd_host; the host tensors it made are appended to `keep`, which the caller
    holds until the stream is synchronised (the copies read them asynchronously)."""
    p = skv.params_for(w, DEV)
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    qh, kh, vh = pin(q), pin(k), pin(v)
    out = pin(torch.empty(w.total_q, w.H, w.d_v, dtype=q.dtype))
    lse = pin(torch.empty(w.H, w.total_q, dtype=torch.float32)) if with_lse else None
    if buf is None:
        buf = torch.empty(skv.sk_host_buffer_bytes(p, DT[w.dtype], with_lse), dtype=torch.uint8,
                          device=DEV)
    skv.sk_attn_fwd_host(p, qh, kh, vh, out, lse, buf, stream=stream)
    if keep is not None:
        keep.extend([qh, kh, vh, buf, p])
    return out, lse


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_host_entry_matches_device_entry_and_oracle(w):
    q, k, v = w.make_inputs("cpu")
    keep = []
    out, lse = _host_run(w, q, k, v, keep=keep)
    torch.cuda.synchronize()
    ref_out, ref_lse, _ = H.run_fwd(w, q.to(DEV), k.to(DEV), v.to(DEV), DEV)
    assert torch.equal(out, ref_out.cpu()) and torch.equal(lse, ref_lse.cpu())
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, w.dtype, "host entry")
    # pageable host memory and no LSE give the same output
    out2, _ = _host_run(w, q, k, v, pinned=False, with_lse=False, keep=keep)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_host_entry_dense_layout():
    w = wl.Workload("dense", H=3, seqlens_q=(200, 200), seqlens_k=(700, 700), d_qk=128, d_v=128,
                    dtype="bf16", seed=65, n_per_block=64, split_kv=3, mask=wl.MASK_CAUSAL)
    q, k, v = w.make_inputs("cpu")
    keep = []
    out_packed, lse_packed = _host_run(w, q, k, v, keep=keep)
    torch.cuda.synchronize()
    p = skv.params_for(w, DEV)
    p.cu_seqlens_q = p.cu_seqlens_k = None
    qb, kb, vb = (t.view(2, -1, 3, 128).pin_memory() for t in (q, k, v))
    out = torch.empty(2, 200, 3, 128, dtype=q.dtype).pin_memory()
    lse = torch.empty(3, 400, dtype=torch.float32).pin_memory()
    buf = torch.empty(skv.sk_host_buffer_bytes(p, skv.SK_BF16, True), dtype=torch.uint8, device=DEV)
    skv.sk_attn_fwd_host(p, qb, kb, vb, out, lse, buf)
    torch.cuda.synchronize()
    assert torch.equal(out.view_as(out_packed), out_packed) and torch.equal(lse, lse_packed)


def test_host_entry_on_two_streams():
    """Two calls in flight on two streams with two device buffers, as the overlapped form runs:
    each matches the device entry point."""
    w = CASES[0]
    q, k, v = w.make_inputs("cpu")
    q2, k2, v2 = w.with_(seed=66).make_inputs("cpu")
    p = skv.params_for(w, DEV)
    nbytes = skv.sk_host_buffer_bytes(p, skv.SK_BF16, True)
    bufs = [torch.empty(nbytes, dtype=torch.uint8, device=DEV) for _ in range(2)]
    streams = [torch.cuda.Stream(device=DEV) for _ in range(2)]
    keep = []
    a = _host_run(w, q, k, v, stream=streams[0], buf=bufs[0], keep=keep)
    b = _host_run(w, q2, k2, v2, stream=streams[1], buf=bufs[1], keep=keep)
    torch.cuda.synchronize()
    for (out, lse), (qq, kk, vv) in ((a, (q, k, v)), (b, (q2, k2, v2))):
        ref_out, ref_lse, _ = H.run_fwd(w, qq.to(DEV), kk.to(DEV), vv.to(DEV), DEV)
        assert torch.equal(out, ref_out.cpu()) and torch.equal(lse, ref_lse.cpu())
