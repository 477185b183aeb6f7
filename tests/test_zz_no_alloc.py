"""sk_attn_fwd_static, the allocation-free entry point, checked against sk_attn_fwd.

Some users of this library cannot allocate device memory where they run attention:
their device memory is planned once up front (a serving loop that must not allocate
per request), or a host framework owns every allocation and gives plugins no
allocator. They cannot pass sk_attn_fwd a workspace, so sk_attn_fwd_static keeps the
split partials in a fixed scratch array inside the library instead.

Both entry points are called through the C ABI on the same inputs; two static calls
in a row (with different inputs, so the second one runs over the scratch the first
one left behind) must each match the workspace entry point within the tolerances of
the parity tests. The file is named to be collected last, so that a run stopping at
the first failure has run every other test already.
"""
from __future__ import annotations

import pytest
import torch

import split_kv_attention_flash_gb300 as skv
from split_kv_attention_flash_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL_O = {"bf16": 2e-2, "f16": 2e-2, "f32": 1e-5}
TOL_LSE = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from split_kv_attention_flash_gb300 import _build
    _build.build()
    skv.lib()


CASES = [
    wl.Workload("decode-like", H=8, seqlens_q=(1,) * 6, seqlens_k=(5000, 17, 900, 0, 3000, 64),
                d_qk=128, d_v=128, dtype="bf16", seed=21, n_per_block=128, split_kv=8),
    wl.Workload("prefill", H=4, seqlens_q=(700, 333), seqlens_k=(9000, 4000), d_qk=192, d_v=128,
                dtype="bf16", seed=22, n_per_block=128, split_kv=3, mask=wl.MASK_PREFIX_CAUSAL,
                prefix_offset=5000),
    wl.Workload("f32 causal", H=2, seqlens_q=(64, 90), seqlens_k=(256, 300), d_qk=64, d_v=64,
                dtype="f32", seed=23, n_per_block=32, split_kv=4, mask=wl.MASK_CAUSAL),
    # the merge fused into the tensor-core kernel (256-row M blocks): its tickets live in
    # the shared scratch too, are cleared by every call and counted up again
    wl.Workload("fused merge", H=3, seqlens_q=(600, 257, 40), seqlens_k=(5000, 1300, 900),
                d_qk=128, d_v=128, dtype="bf16", seed=24, n_per_block=128, split_kv=4,
                mask=wl.MASK_PREFIX_CAUSAL, prefix_offset=700, extra={"fuse_combine": 1}),
]


def _params(w):
    return skv.params_for(w, DEV, fuse_combine=w.extra.get("fuse_combine", 0))


def _run(w, seed, static):
    q, k, v = w.with_(seed=seed).make_inputs(DEV)
    p = _params(w)
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=q.dtype, device=DEV)
    lse = torch.empty(w.H, w.total_q, dtype=torch.float32, device=DEV)
    if static:
        skv.sk_attn_fwd_static(p, q, k, v, out, lse)
    else:
        ws = torch.empty(max(skv.sk_workspace_bytes(p), 1), dtype=torch.uint8, device=DEV)
        skv.sk_attn_fwd(p, q, k, v, out, lse, ws)
    torch.cuda.synchronize()
    return out.float(), lse


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_static_entry_matches_workspace_entry_on_two_calls(w):
    assert skv.sk_workspace_bytes(_params(w)) <= skv.SK_STATIC_SCRATCH_BYTES
    for seed in (w.seed, w.seed + 100):          # two calls in a row, different inputs
        ref_o, ref_l = _run(w, seed, static=False)
        got_o, got_l = _run(w, seed, static=True)
        assert not torch.isnan(got_o).any() and not torch.isnan(got_l).any()
        assert (got_o - ref_o).abs().max().item() <= TOL_O[w.dtype]
        inf = torch.isneginf(ref_l)
        assert torch.equal(torch.isneginf(got_l), inf)
        assert (got_l[~inf] - ref_l[~inf]).abs().max().item() <= TOL_LSE


def test_static_entry_rejects_problems_above_its_scratch():
    w = wl.TARGET_SHAPE.with_(split_kv=8)
    p = skv.params_for(w, DEV)
    assert skv.sk_workspace_bytes(p) > skv.SK_STATIC_SCRATCH_BYTES
    q = torch.empty(w.total_q, w.H, w.d_qk, dtype=torch.bfloat16, device=DEV)
    k = torch.empty(w.total_k, w.H, w.d_qk, dtype=torch.bfloat16, device=DEV)
    v = torch.empty(w.total_k, w.H, w.d_v, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(skv.SplitKVError) as ei:
        skv.sk_attn_fwd_static(p, q, k, v, out)
    assert ei.value.status == 3  # SK_ERR_WORKSPACE


def test_static_entry_allocates_no_device_memory():
    """After a first call (which looks up the scratch array and loads the kernels), a call
    leaves both torch's allocator and the device's free memory unchanged."""
    w = CASES[1]
    q, k, v = w.make_inputs(DEV)
    p = _params(w)
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=q.dtype, device=DEV)
    lse = torch.empty(w.H, w.total_q, dtype=torch.float32, device=DEV)
    skv.sk_attn_fwd_static(p, q, k, v, out, lse)
    torch.cuda.synchronize()
    allocated = torch.cuda.memory_allocated(DEV)
    free_before = torch.cuda.mem_get_info(DEV)[0]
    skv.sk_attn_fwd_static(p, q, k, v, out, lse)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(DEV)[0] == free_before
    assert torch.cuda.memory_allocated(DEV) == allocated
