"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Small problems (several M blocks and key tiles, ragged tails, every mask, every
storage type and head-dim pair) are compared element by element; the full-size
workloads are compared on sampled rows (all heads; per sequence the first and
last rows plus seeded random rows). Split counts are compared bit-exactly.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import split_kv_attention_flash_gb300 as skv
from split_kv_attention_flash_gb300 import workloads as wl
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from split_kv_attention_flash_gb300 import _build
    _build.build()
    skv.lib()


def _small(dtype, dqk, dv, mask=wl.MASK_NONE, po=0, lvi=-1, bn=64, S=3, seed=0,
           sq=(300, 1, 77, 256), sk=(1000, 5, 0, 513), window=-1, used=None):
    name = f"small {dtype} {dqk}/{dv} mask{mask} po{po} lvi{lvi} S{S}"
    if window >= 0:
        name += f" window{window}"
    if used is not None:
        name += " padded"
    return wl.Workload(name, H=2, seqlens_q=sq, seqlens_k=sk, d_qk=dqk, d_v=dv, dtype=dtype,
                       seed=seed, n_per_block=bn, split_kv=S, mask=mask, prefix_offset=po,
                       last_valid_kv_index=lvi, window_left=window, seqused_k=used)


SMALL = [
    wl.TINY_CAUSAL,
    _small("bf16", 128, 128),
    _small("bf16", 192, 128, mask=wl.MASK_CAUSAL, S=4, bn=128),
    _small("f16", 64, 64, mask=wl.MASK_PREFIX_CAUSAL, po=40, lvi=700, S=5, bn=32),
    _small("f16", 128, 128, mask=wl.MASK_PREFIX_CAUSAL, po=-100, S=2, bn=16),
    _small("f32", 192, 128, mask=wl.MASK_CAUSAL, lvi=200, S=8, bn=48),
    _small("bf16", 64, 64, S=1),
    _small("bf16", 192, 128, S=7, bn=128, sq=(1, 1, 1), sk=(3000, 17, 0)),
    # sliding windows and padded key slots (per-sequence used counts)
    _small("bf16", 192, 128, mask=wl.MASK_CAUSAL, S=4, bn=128, window=300),
    _small("f16", 128, 128, mask=wl.MASK_PREFIX_CAUSAL, po=500, S=3, bn=64, window=100,
           used=(900, 5, 0, 400)),
    _small("bf16", 128, 128, S=5, bn=128, sq=(1, 1, 1, 2), sk=(3000, 70, 500, 900),
           used=(2500, 80, 3, 0)),
    _small("bf16", 64, 64, mask=wl.MASK_PREFIX_CAUSAL, po=2000, S=6, bn=128, window=700,
           sq=(1, 3, 16), sk=(3000, 2500, 2100)),
    _small("f32", 128, 128, mask=wl.MASK_CAUSAL, S=3, bn=32, window=40, used=(800, 5, 0, 300)),
    # unmasked, two or more M blocks, including blocks past a sequence's end, padded key
    # slots and lastValid
    _small("f16", 192, 128, S=2, bn=128, sq=(600, 257, 3), sk=(900, 1300, 40)),
    _small("bf16", 192, 128, S=3, bn=128, sq=(520, 300), sk=(2000, 700), used=(1800, 1)),
    _small("f16", 128, 128, lvi=600, S=4, bn=64, sq=(700,), sk=(1500,)),
    # at most 128 queries per sequence: the tensor-core kernel splits each block's key
    # tiles between its two halves (odd and even tile counts, one-tile splits, masks,
    # windows, padded key slots, each head dim)
    _small("bf16", 192, 128, mask=wl.MASK_PREFIX_CAUSAL, po=1000, S=3, bn=128,
           sq=(128, 100, 2, 77), sk=(3000, 1500, 700, 129)),
    _small("f16", 128, 128, lvi=900, S=4, bn=64, sq=(64, 128, 5), sk=(2000, 900, 3000)),
    _small("bf16", 128, 128, mask=wl.MASK_PREFIX_CAUSAL, po=1500, S=2, bn=128, window=300,
           sq=(120, 128), sk=(2000, 1700), used=(1900, 1650)),
    _small("bf16", 64, 64, S=5, bn=128, sq=(33, 2), sk=(5000, 4000)),
    # S = 1 writes the output directly
    _small("bf16", 192, 128, S=1, bn=128, sq=(513, 40), sk=(1000, 3000)),
]


# limits and degenerate shapes: the largest split count, single-key and 256-key partition
# tiles, many short sequences (some without queries or keys), many heads, lastValid = 0,
# a one-key sliding window
LIMITS = [
    _small("bf16", 128, 128, mask=wl.MASK_CAUSAL, S=32, bn=16, sq=(300,), sk=(4000,)),
    _small("bf16", 64, 64, mask=wl.MASK_CAUSAL, S=5, bn=1, sq=(100, 40), sk=(300, 57)),
    _small("f16", 192, 128, S=3, bn=256, sq=(520,), sk=(3000,)),
    wl.Workload("many short sequences", H=4,
                seqlens_q=tuple(int(x) for x in np.random.default_rng(5).integers(0, 41, 64)),
                seqlens_k=tuple(int(x) for x in np.random.default_rng(6).integers(0, 501, 64)),
                d_qk=128, d_v=128, dtype="bf16", seed=5, n_per_block=16, split_kv=4,
                mask=wl.MASK_PREFIX_CAUSAL, prefix_offset=20),
    wl.Workload("many heads", H=64, seqlens_q=(260,), seqlens_k=(700,), d_qk=64, d_v=64,
                dtype="bf16", seed=7, n_per_block=128, split_kv=2),
    _small("bf16", 128, 128, S=3, bn=64, sq=(0, 70, 0, 300), sk=(50, 0, 900, 400)),
    _small("bf16", 192, 128, S=4, bn=128, lvi=0, sq=(50, 300), sk=(1000, 10)),
    _small("f16", 128, 128, mask=wl.MASK_PREFIX_CAUSAL, po=100, S=3, bn=64, window=0,
           sq=(300, 17), sk=(800, 200)),
]


def _inputs(w):
    q, k, v = w.make_inputs("cpu")
    return (q, k, v), (q.to(DEV), k.to(DEV), v.to(DEV))


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_counts_bit_exact_small(w):
    S = H.resolved_split(w, DEV)
    p = skv.params_for(w, DEV, split_kv=S)
    counts = torch.full((w.total_q,), -7, dtype=torch.int32, device=DEV)
    skv.sk_valid_split_counts(p, counts)
    ref = oracle.split_counts(H.oracle_problem(w, S))
    assert np.array_equal(counts.cpu().numpy(), ref)


def test_counts_bit_exact_sweep():
    rng = np.random.default_rng(123)
    for _ in range(150):
        B = int(rng.integers(1, 4))
        sq = tuple(int(x) for x in rng.integers(1, 70, B))
        sk = tuple(int(x) for x in rng.integers(0, 300, B))
        mask = int(rng.integers(0, 3))
        po = int(rng.integers(-80, 300)) if mask == wl.MASK_PREFIX_CAUSAL else 0
        w = wl.Workload("sweep", H=1, seqlens_q=sq, seqlens_k=sk, d_qk=64, d_v=64, dtype="bf16",
                        seed=0, n_per_block=int(rng.choice([1, 16, 32, 48, 128])),
                        split_kv=int(rng.integers(1, 33)), mask=mask, prefix_offset=po,
                        last_valid_kv_index=int(rng.choice([-1, 0, 50, 1000])))
        p = skv.params_for(w, DEV)
        counts = torch.empty(w.total_q, dtype=torch.int32, device=DEV)
        skv.sk_valid_split_counts(p, counts)
        ref = oracle.split_counts(H.oracle_problem(w, w.split_kv))
        assert np.array_equal(counts.cpu().numpy(), ref), w


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_partials_match_oracle_small(w):
    (q, k, v), (qd, kd, vd) = _inputs(w)
    S = H.resolved_split(w, DEV)
    o_part, l_part, _ = H.run_partials(w, qd, kd, vd, DEV, S)
    ref_o, ref_l = oracle.partials(H.oracle_problem(w, S), q, k, v)      # [n, H, S, dv]
    got_o = o_part.permute(2, 0, 1, 3).cpu().numpy()
    got_l = l_part.permute(2, 0, 1).cpu().numpy()
    H.assert_close(got_o, got_l, ref_o, ref_l, w.dtype, "partials")
    # empty (row, split) pairs: exact zero output and -inf LSE
    empty = np.isneginf(ref_l)
    assert (got_o[empty] == 0).all() and np.isneginf(got_l[empty]).all()


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_forward_matches_oracle_small(w):
    (q, k, v), (qd, kd, vd) = _inputs(w)
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    out, lse, p = H.run_fwd(w, qd, kd, vd, DEV)
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, w.dtype, "forward")
    # without an LSE output the output is identical
    out2, _, _ = H.run_fwd(w, qd, kd, vd, DEV, with_lse=False)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("w", LIMITS, ids=lambda w: w.name)
def test_limits_match_oracle(w):
    (q, k, v), (qd, kd, vd) = _inputs(w)
    S = H.resolved_split(w, DEV)
    p = skv.params_for(w, DEV, split_kv=S)
    counts = torch.full((w.total_q,), -7, dtype=torch.int32, device=DEV)
    skv.sk_valid_split_counts(p, counts)
    assert np.array_equal(counts.cpu().numpy(), oracle.split_counts(H.oracle_problem(w, S)))
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    out, lse, _ = H.run_fwd(w, qd, kd, vd, DEV)
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, w.dtype, "forward")


@pytest.mark.parametrize("w", [
    _small("bf16", 192, 128, S=3, bn=128, sq=(520,), sk=(3000,)),
    _small("f16", 128, 128, mask=wl.MASK_CAUSAL, S=4, bn=64, sq=(300,), sk=(900,)),
], ids=lambda w: w.name)
def test_large_logits_match_oracle(w):
    """Q and K scaled by 6 (scores of a few hundred): the running max jumps within and across
    key tiles, the lazy rescale of O fires, and a few keys dominate each row."""
    (q, k, v), _ = _inputs(w)
    q, k = (t.float().mul(6.0).to(t.dtype) for t in (q, k))
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    assert ref_l.max() > 100.0
    out, lse, _ = H.run_fwd(w, qd, kd, vd, DEV)
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, w.dtype, "forward")


@pytest.mark.parametrize("dtype,mask,po,sq", [
    ("bf16", wl.MASK_NONE, 0, (1, 2, 3, 16, 8, 5)),
    ("f16", wl.MASK_PREFIX_CAUSAL, 700, (1, 2, 3, 16, 8, 5)),
    ("bf16", wl.MASK_PREFIX_CAUSAL, 500, (1, 1, 1, 1, 1, 1)),
])
def test_decode_kernel_with_several_queries(dtype, mask, po, sq):
    """Up to 16 queries per sequence with an M block of 64 rows: the tensor-core kernel
    (256-row M blocks) does not apply, so the CUDA-core decode kernel takes every query
    count it is templated on (1, 2, 4, 8, 16)."""
    w = _small(dtype, 128, 128, mask=mask, po=po, S=3, bn=64, sq=sq,
               sk=(900, 40, 0, 1000, 777, 300))
    (q, k, v), (qd, kd, vd) = _inputs(w)
    bm = 64
    p = skv.params_for(w, DEV, split_kv=3, block_m=bm)
    assert skv.sk_partial_kernel_name(p, qd, kd, vd) == "partial_decode"
    o_part = torch.empty(w.H, 3, w.total_q, w.d_v, dtype=torch.float32, device=DEV)
    l_part = torch.empty(w.H, 3, w.total_q, dtype=torch.float32, device=DEV)
    skv.sk_attn_partial_fwd(p, qd, kd, vd, o_part, l_part)
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=qd.dtype, device=DEV)
    lse = torch.empty(w.H, w.total_q, dtype=torch.float32, device=DEV)
    ws = torch.empty(max(skv.sk_workspace_bytes(p), 1), dtype=torch.uint8, device=DEV)
    skv.sk_attn_fwd(p, qd, kd, vd, out, lse, ws)
    torch.cuda.synchronize()
    ref_po, ref_pl = oracle.partials(H.oracle_problem(w, 3, block_m=bm), q, k, v)
    H.assert_close(o_part.permute(2, 0, 1, 3).cpu().numpy(), l_part.permute(2, 0, 1).cpu().numpy(),
                   ref_po, ref_pl, w.dtype, "partials")
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, w.dtype, "forward")


@pytest.mark.parametrize("B,S", [(8, 4), (64, 4), (65, 4), (130, 2)])
def test_single_query_on_the_tensor_cores(B, S):
    """One query per sequence runs on the tensor-core kernel's single-block form: units taken
    longest first up to 256 (sequence, split) units, in index order beyond; both match the
    oracle, for the partials and for the output written directly at split 1."""
    kernel = "partial_tc"
    rng = np.random.default_rng(B)
    w = _small("bf16", 128, 128, S=S, bn=128, sq=(1,) * B,
               sk=tuple(int(x) for x in rng.integers(0, 700, B)))
    (q, k, v), (qd, kd, vd) = _inputs(w)
    p = skv.params_for(w, DEV, split_kv=S)
    assert skv.sk_partial_kernel_name(p, qd, kd, vd) == kernel
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    for split in (S, 1):
        out, lse, _ = H.run_fwd(w, qd, kd, vd, DEV, split_kv=split)
        H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, w.dtype, f"forward S={split}")
    o_part, l_part, _ = H.run_partials(w, qd, kd, vd, DEV, S)
    ref_po, ref_pl = oracle.partials(H.oracle_problem(w, S), q, k, v)
    H.assert_close(o_part.permute(2, 0, 1, 3).cpu().numpy(), l_part.permute(2, 0, 1).cpu().numpy(),
                   ref_po, ref_pl, w.dtype, "partials")


def test_long_single_sequence_sampled():
    """One sequence of 262144 keys (well past the workloads' longest), sampled rows."""
    w = wl.Workload("long single sequence", H=2, seqlens_q=(512,), seqlens_k=(262144,), d_qk=128,
                    d_v=128, dtype="bf16", seed=8, n_per_block=128, split_kv=0, value_scale=0.5)
    (q, k, v), (qd, kd, vd) = _inputs(w)
    out, lse, p = H.run_fwd(w, qd, kd, vd, DEV)
    rows = H.sample_rows(w, head=32, tail=32, rand=32)
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v, rows=rows)
    H.assert_close(H.to_np(out, rows), H.lse_np(lse, rows), ref_o, ref_l, w.dtype, "forward")


@pytest.mark.parametrize("w", SMALL[:4], ids=lambda w: w.name)
def test_split_one_direct_equals_partial_plus_combine(w):
    (_, _, _), (qd, kd, vd) = _inputs(w)
    out, lse, p = H.run_fwd(w, qd, kd, vd, DEV, split_kv=1)
    o_part, l_part, p1 = H.run_partials(w, qd, kd, vd, DEV, 1)
    counts = torch.empty(w.total_q, dtype=torch.int32, device=DEV)
    skv.sk_valid_split_counts(p1, counts)
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    skv.sk_combine(p1, o_part, l_part, counts, out2, lse2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    assert torch.equal(lse, lse2)


@pytest.mark.parametrize("w", SMALL[1:4], ids=lambda w: w.name)
def test_combine_never_reads_invalid_splits(w):
    (_, _, _), (qd, kd, vd) = _inputs(w)
    S = H.resolved_split(w, DEV)
    o_part, l_part, p = H.run_partials(w, qd, kd, vd, DEV, S)
    counts = torch.empty(w.total_q, dtype=torch.int32, device=DEV)
    skv.sk_valid_split_counts(p, counts)
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=qd.dtype, device=DEV)
    lse = torch.empty(w.H, w.total_q, dtype=torch.float32, device=DEV)
    skv.sk_combine(p, o_part, l_part, counts, out, lse)
    s_idx = torch.arange(S, device=DEV)[None, :, None]
    invalid = s_idx >= counts[None, None, :]                       # [1, S, total_q]
    o_bad = o_part.masked_fill(invalid[..., None], float("nan"))
    l_bad = l_part.masked_fill(invalid, float("nan"))
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    skv.sk_combine(p, o_bad, l_bad, counts, out2, lse2)
    torch.cuda.synchronize()
    assert invalid.any() or S == 1
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    assert not torch.isnan(out2.float()).any()


@pytest.mark.parametrize("mask,sq,S", [(wl.MASK_CAUSAL, 130, 3), (wl.MASK_NONE, 300, 3),
                                       (wl.MASK_NONE, 1, 3), (wl.MASK_NONE, 1, 1),
                                       (wl.MASK_PREFIX_CAUSAL, 100, 1)])
def test_dense_layout_equals_varlen(mask, sq, S):
    """[B, seq, H, D] tensors without cu_seqlens give the packed layout's results bit for bit
    (two-tile and single-block forms, partials and direct output)."""
    w = wl.Workload("dense", H=3, seqlens_q=(sq, sq), seqlens_k=(400, 400), d_qk=128, d_v=128,
                    dtype="bf16", seed=9, n_per_block=64, split_kv=S, mask=mask,
                    prefix_offset=300 if mask == wl.MASK_PREFIX_CAUSAL else 0)
    (_, _, _), (qd, kd, vd) = _inputs(w)
    out, lse, _ = H.run_fwd(w, qd, kd, vd, DEV)
    p = skv.params_for(w, DEV)
    p.cu_seqlens_q = p.cu_seqlens_k = None
    qb = qd.view(2, sq, 3, 128)
    kb, vb = kd.view(2, 400, 3, 128), vd.view(2, 400, 3, 128)
    outb = torch.empty(2, sq, 3, 128, dtype=qd.dtype, device=DEV)
    lseb = torch.empty(3, 2 * sq, dtype=torch.float32, device=DEV)
    ws = torch.empty(skv.sk_workspace_bytes(p), dtype=torch.uint8, device=DEV)
    skv.sk_attn_fwd(p, qb, kb, vb, outb, lseb, ws)
    torch.cuda.synchronize()
    assert torch.equal(outb.view_as(out), out) and torch.equal(lseb, lse)


@pytest.mark.parametrize("mask", [wl.MASK_CAUSAL, wl.MASK_NONE])
def test_strided_heads_and_rows(mask):
    """Q/K/V as views into wider buffers (row stride > H * d)."""
    w = _small("bf16", 128, 128, mask=mask, S=3)
    (q, k, v), (qd, kd, vd) = _inputs(w)
    pad = 8
    def widen(t):
        big = torch.zeros(t.shape[0], t.shape[1] + 1, t.shape[2] + pad, dtype=t.dtype, device=DEV)
        big[:, 1:, pad:] = t
        return big[:, 1:, pad:]
    out_ref, lse_ref, p = H.run_fwd(w, qd, kd, vd, DEV)
    qs, ks, vs = widen(qd), widen(kd), widen(vd)
    out = widen(torch.empty_like(out_ref))
    lse = torch.empty_like(lse_ref)
    ws = torch.empty(skv.sk_workspace_bytes(p), dtype=torch.uint8, device=DEV)
    skv.sk_attn_fwd(p, qs, ks, vs, out, lse, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref)


def test_empty_keys_give_zero_and_neg_inf():
    for S in (1, 4):
        w = wl.Workload("no keys", H=2, seqlens_q=(5, 9), seqlens_k=(0, 0), d_qk=128, d_v=128,
                        dtype="bf16", seed=1, n_per_block=128, split_kv=S)
        (_, _, _), (qd, kd, vd) = _inputs(w)
        kd = torch.zeros(1, 2, 128, dtype=qd.dtype, device=DEV)   # a real (unused) buffer
        vd = torch.zeros(1, 2, 128, dtype=qd.dtype, device=DEV)
        out, lse, _ = H.run_fwd(w, qd, kd, vd, DEV)
        assert (out == 0).all() and torch.isneginf(lse).all()


def test_graph_capture_and_replay():
    w = _small("bf16", 192, 128, mask=wl.MASK_CAUSAL, S=4, bn=128)
    (q, k, v), (qd, kd, vd) = _inputs(w)
    out_ref, lse_ref, p = H.run_fwd(w, qd, kd, vd, DEV)
    out = torch.empty_like(out_ref)
    lse = torch.empty_like(lse_ref)
    ws = torch.empty(skv.sk_workspace_bytes(p), dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        skv.sk_attn_fwd(p, qd, kd, vd, out, lse, ws, stream=s)   # warm up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g):
        skv.sk_attn_fwd(p, qd, kd, vd, out, lse, ws)
    out.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref)
    # new inputs in the same buffers are picked up by the replay
    qd.mul_(0.5)
    out_new, lse_new, _ = H.run_fwd(w, qd, kd, vd, DEV)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, out_new) and torch.equal(lse, lse_new)


# ------------------------------------------------------------ full-size configs

def _sampled_check(w, splits, rows_kw=None, seq_subset=None):
    """Run the full-size workload for each split count and compare sampled rows.

    With seq_subset, the oracle sees only those sequences (their Q/K/V rows copied
    out), which keeps host memory small for the decode workload."""
    q, k, v = w.make_inputs(DEV)
    seqs = list(range(w.B)) if seq_subset is None else list(seq_subset)
    sub = w.with_(seqlens_q=tuple(w.seqlens_q[b] for b in seqs),
                  seqlens_k=tuple(w.seqlens_k[b] for b in seqs))
    def gather(t, cu):
        return torch.cat([t[cu[b]:cu[b + 1]] for b in seqs]).cpu()
    qc, kc, vc = gather(q, w.cu_seqlens_q), gather(k, w.cu_seqlens_k), gather(v, w.cu_seqlens_k)
    sub_rows = H.sample_rows(sub, **(rows_kw or {}))
    # packed row of the subset -> packed row of the full problem
    full_of_sub = np.concatenate([np.arange(w.cu_seqlens_q[b], w.cu_seqlens_q[b + 1])
                                  for b in seqs]).astype(np.int64)
    rows = full_of_sub[sub_rows]
    ref_o, ref_l = oracle.attention(H.oracle_problem(sub, 1), qc, kc, vc, rows=sub_rows)
    del qc, kc, vc
    for S in splits:
        out, lse, p = H.run_fwd(w, q, k, v, DEV, split_kv=S)
        H.assert_close(H.to_np(out, rows), H.lse_np(lse, rows), ref_o, ref_l, w.dtype,
                       f"{w.name} S={S}")
        S_res = skv.sk_auto_split_kv(p)
        counts = torch.empty(w.total_q, dtype=torch.int32, device=DEV)
        skv.sk_valid_split_counts(p, counts)
        ref_c = oracle.split_counts(H.oracle_problem(w, S_res))
        assert np.array_equal(counts.cpu().numpy(), ref_c)
        del out, lse


def test_config_noncausal_bf16_full():
    _sampled_check(wl.NONCAUSAL_BF16, [1, 2, 4, 8])


@pytest.mark.parametrize("mask,po", [(wl.MASK_CAUSAL, 0), (wl.MASK_PREFIX_CAUSAL, 2048),
                                     (wl.MASK_PREFIX_CAUSAL, -256)])
def test_config_masked_f16_full(mask, po):
    _sampled_check(wl.MASKED_F16.with_(mask=mask, prefix_offset=po), [4])


def test_config_long_varlen_full():
    w = wl.LONG_VARLEN
    assert H.resolved_split(w, DEV) == 3
    _sampled_check(w, [0, 2, 3, 4, 5, 6, 7, 8], rows_kw=dict(head=16, tail=16, rand=16))


def test_ragged_causal_prefill_over_many_waves():
    """Three ragged sequences under a causal mask with far more CTAs than SMs (11 M blocks x
    16 heads x 9 units): the tensor-core kernel takes the (sequence, split) units longest
    first and each sequence's M blocks last-first. Sampled rows of every sequence against the
    oracle, at the automatic split and at 3, plus the split counts bit for bit."""
    w = wl.Workload("ragged causal prefill", H=16, seqlens_q=(1500, 700, 2600),
                    seqlens_k=(1500, 700, 2600), d_qk=192, d_v=128, dtype="bf16", seed=71,
                    n_per_block=128, split_kv=3, mask=wl.MASK_CAUSAL)
    q, k, v = w.make_inputs(DEV)
    assert skv.sk_partial_kernel_name(skv.params_for(w, DEV), q, k, v) == "partial_tc"
    del q, k, v
    _sampled_check(w, [0, 3], rows_kw=dict(head=32, tail=32, rand=64))


def test_target_shape_full():
    """The benchmark's default workload in the launch it times: automatic split (3)."""
    w = wl.TARGET_SHAPE
    assert H.resolved_split(w, DEV) == 3
    _sampled_check(w, [0, 3], rows_kw=dict(head=32, tail=32, rand=64))


def test_config_decode_full():
    w = wl.DECODE
    _sampled_check(w, [0, 1, 2, 4, 8, 16, 32], seq_subset=[0, 7, 19, 31])


def test_config_target_d128_full():
    w = wl.TARGET_D128
    assert H.resolved_split(w, DEV) == 3
    _sampled_check(w, [0], rows_kw=dict(head=32, tail=32, rand=64))


def test_config_window_full():
    """The sliding-window workload: the window hides split 0 of 3 from the deepest rows, so
    auto keeps it unsplit; forced splits leave the leading splits of those rows empty."""
    w = wl.WINDOW
    assert H.resolved_split(w, DEV) == 1
    _sampled_check(w, [0, 2, 3], rows_kw=dict(head=32, tail=32, rand=64))


def test_config_decode_mq_full():
    """Eight queries per sequence go to the tensor-core kernel (auto: 3 splits)."""
    w = wl.DECODE_MQ
    assert H.resolved_split(w, DEV) == 3
    _sampled_check(w, [0, 1, 4], seq_subset=[0, 7, 19, 31])


def test_config_decode_small_full():
    w = wl.DECODE_SMALL
    assert H.resolved_split(w, DEV) == 1
    _sampled_check(w, [0, 2], seq_subset=[0, 13, 31])


@pytest.mark.parametrize("w", [SMALL[1], SMALL[2], SMALL[4], SMALL[-1]], ids=lambda w: w.name)
def test_fused_merge_matches_separate_combine(w):
    """sk_attn_fwd with fuse_combine = 1 (the tensor-core kernel merges in the last CTA of
    each M block) against the default one-call path and the three separate calls."""
    (_, _, _), (qd, kd, vd) = _inputs(w)
    S = H.resolved_split(w, DEV)
    out, lse, _ = H.run_fwd(w, qd, kd, vd, DEV, split_kv=S, fuse_combine=1)
    ref, ref_lse, _ = H.run_fwd(w, qd, kd, vd, DEV, split_kv=S)
    o_part, l_part, p = H.run_partials(w, qd, kd, vd, DEV, S)
    counts = torch.empty(w.total_q, dtype=torch.int32, device=DEV)
    skv.sk_valid_split_counts(p, counts)
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    skv.sk_combine(p, o_part, l_part, counts, out2, lse2)
    torch.cuda.synchronize()
    for o, l in ((out2, lse2), (ref, ref_lse)):
        assert (out.float() - o.float()).abs().max().item() <= H.TOL_O[w.dtype]
        inf = torch.isneginf(l)
        assert torch.equal(torch.isneginf(lse), inf)
        assert (lse[~inf] - l[~inf]).abs().max().item() <= 1e-5
    # a second call reuses the workspace: every call zeroes the tickets
    out3, lse3, _ = H.run_fwd(w, qd, kd, vd, DEV, split_kv=S, fuse_combine=1)
    assert torch.equal(out, out3) and torch.equal(lse, lse3)


@pytest.mark.parametrize("w", [wl.TINY_CAUSAL, SMALL[3], SMALL[4]], ids=lambda w: w.name)
def test_combine_never_reads_partition_empty_splits(w):
    """Splits the M-block partition leaves empty may hold anything (sk_attn_fwd does not
    write them): poisoning them with NaN changes nothing."""
    (_, _, _), (qd, kd, vd) = _inputs(w)
    S = H.resolved_split(w, DEV)
    o_part, l_part, p = H.run_partials(w, qd, kd, vd, DEV, S)
    counts = torch.empty(w.total_q, dtype=torch.int32, device=DEV)
    skv.sk_valid_split_counts(p, counts)
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=qd.dtype, device=DEV)
    lse = torch.empty(w.H, w.total_q, dtype=torch.float32, device=DEV)
    skv.sk_combine(p, o_part, l_part, counts, out, lse)
    kb, ke = oracle.split_ranges(H.oracle_problem(w, S))                 # [total_q, S]
    empty = torch.from_numpy(ke <= kb).to(DEV).T                          # [S, total_q]
    assert empty.any()
    o_bad = o_part.masked_fill(empty[None, :, :, None], float("nan"))
    l_bad = l_part.masked_fill(empty[None], float("nan"))
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    skv.sk_combine(p, o_bad, l_bad, counts, out2, lse2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


# ------------------------------------------- every public path against the oracle
#
# "Recombine fully masked split-KV attention partials on the host", Technical details:
# the NaN-safe f32 merge over the splits s < count. Besides sk_attn_fwd (above), the
# library exposes two more ways of getting the merged output; each is compared here with
# the f64 oracle, element by element, at the stated tolerances.

def _three_call(w, qd, kd, vd, S, with_lse=True):
    """sk_attn_partial_fwd -> sk_valid_split_counts -> sk_combine with the caller's counts."""
    o_part, l_part, p = H.run_partials(w, qd, kd, vd, DEV, S)
    counts = torch.full((w.total_q,), -7, dtype=torch.int32, device=DEV)
    skv.sk_valid_split_counts(p, counts)
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=qd.dtype, device=DEV)
    lse = torch.empty(w.H, w.total_q, dtype=torch.float32, device=DEV) if with_lse else None
    skv.sk_combine(p, o_part, l_part, counts, out, lse)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("w", SMALL + LIMITS, ids=lambda w: w.name)
def test_three_call_path_matches_oracle(w):
    """The standalone public path, with the counts array the caller got from
    sk_valid_split_counts, against unsplit attention; without an LSE output the output is
    identical."""
    (q, k, v), (qd, kd, vd) = _inputs(w)
    S = H.resolved_split(w, DEV)
    out, lse = _three_call(w, qd, kd, vd, S)
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, w.dtype, f"three calls S={S}")
    out2, _ = _three_call(w, qd, kd, vd, S, with_lse=False)
    assert torch.equal(out, out2)


def _oracle_partials_on_device(prob, q, k, v):
    """The oracle's partials, rounded to f32 (the workspace's type), in the library's
    [H, S, total_q, d_v] / [H, S, total_q] layout, plus the f32 values as f64 arrays."""
    po, pl = oracle.partials(prob, q, k, v)                    # [n, H, S, dv], [n, H, S]
    po32, pl32 = po.astype(np.float32), pl.astype(np.float32)
    o_dev = torch.from_numpy(np.ascontiguousarray(po32.transpose(1, 2, 0, 3))).to(DEV)
    l_dev = torch.from_numpy(np.ascontiguousarray(pl32.transpose(1, 2, 0))).to(DEV)
    return o_dev, l_dev, po32.astype(np.float64), pl32.astype(np.float64)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("S", [1, 2, 3, 5, 8, 9, 16, 32])
def test_combine_of_oracle_partials_matches_oracle_merge(S, dtype):
    """sk_combine alone, fed the oracle's own partials and counts: its output and LSE against
    the oracle's merge of the same f32 values. Covers the bulk-copy form (S <= 8), the
    register-prefetch form (S > 8), fully masked rows (prefix offset < 0, a sequence without
    keys), rows whose count is below S, and splits s >= count filled with NaN, which the
    merge must never read."""
    w = _small(dtype, 128, 128, mask=wl.MASK_PREFIX_CAUSAL, po=-50, S=S, bn=16,
               sq=(300, 40, 0, 7), sk=(900, 600, 30, 0), seed=S)
    q, k, v = w.make_inputs("cpu")
    prob = H.oracle_problem(w, S)
    counts = oracle.split_counts(prob)
    o_dev, l_dev, po, pl = _oracle_partials_on_device(prob, q, k, v)
    invalid = torch.arange(S, device=DEV)[None, :, None] >= torch.from_numpy(counts).to(DEV)[None, None, :]
    o_dev = o_dev.masked_fill(invalid[..., None], float("nan"))
    l_dev = l_dev.masked_fill(invalid, float("nan"))
    p = skv.params_for(w, DEV, split_kv=S)
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=w.torch_dtype, device=DEV)
    lse = torch.empty(w.H, w.total_q, dtype=torch.float32, device=DEV)
    skv.sk_combine(p, o_dev, l_dev, torch.from_numpy(counts).to(DEV), out, lse)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.merge(po, pl, counts)
    assert np.isneginf(ref_l).any() and (counts < S).any() or S == 1
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, dtype, f"combine S={S}")
    # the merge itself runs in f32: before the cast to the storage type it is within f32
    # rounding of the oracle's f64 merge of the same values
    if dtype == "f32":
        assert np.abs(H.to_np(out) - ref_o).max() <= 4e-6


FUSED = [w for w in SMALL + LIMITS if w.dtype != "f32" and 2 <= w.split_kv <= 8]


@pytest.mark.parametrize("w", FUSED, ids=lambda w: w.name)
def test_fused_merge_matches_oracle(w):
    """sk_attn_fwd with fuse_combine = 1: the tensor-core kernel's last CTA of each M block
    merges the splits. Compared with unsplit attention; a second call over the same workspace
    (tickets cleared again) gives identical results, and so does a call without LSE."""
    (q, k, v), (qd, kd, vd) = _inputs(w)
    out, lse, p = H.run_fwd(w, qd, kd, vd, DEV, fuse_combine=1)
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, w.dtype, "fused merge")
    out2, lse2, _ = H.run_fwd(w, qd, kd, vd, DEV, fuse_combine=1)
    out3, _, _ = H.run_fwd(w, qd, kd, vd, DEV, fuse_combine=1, with_lse=False)
    assert torch.equal(out, out2) and torch.equal(lse, lse2) and torch.equal(out, out3)


def test_fused_merge_matches_oracle_full_size():
    """The fused merge on the target shape (automatic split, 3), sampled rows."""
    w = wl.TARGET_SHAPE
    q, k, v = w.make_inputs(DEV)
    rows = H.sample_rows(w, head=32, tail=32, rand=64)
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q.cpu(), k.cpu(), v.cpu(), rows=rows)
    out, lse, _ = H.run_fwd(w, q, k, v, DEV, fuse_combine=1)
    H.assert_close(H.to_np(out, rows), H.lse_np(lse, rows), ref_o, ref_l, w.dtype, "fused target")


# ------------------------------------------------- the persistent tensor-core form
#
# Launches of more (sequence, head, split, M block) units than SMs, each with a few key
# tiles, run on partial_tc_persist: one CTA per SM takes the units in turn. Each case
# below is shaped to land there (checked through sk_partial_kernel_name) and compared with
# the oracle: the partials of sk_attn_partial_fwd (empty splits write 0 / -inf), the
# one-call forward (empty splits write nothing) and the three-call path.

PERSIST = [
    wl.Workload("persist causal bf16 D128 S8", H=8, seqlens_q=(600, 300, 513),
                seqlens_k=(700, 1200, 600), d_qk=128, d_v=128, dtype="bf16", seed=41,
                n_per_block=64, split_kv=8, mask=wl.MASK_CAUSAL),
    wl.Workload("persist prefix window f16 D64 S5", H=12, seqlens_q=(700, 257),
                seqlens_k=(2000, 900), d_qk=64, d_v=64, dtype="f16", seed=42, n_per_block=32,
                split_kv=5, mask=wl.MASK_PREFIX_CAUSAL, prefix_offset=300, window_left=400),
    wl.Workload("persist non-causal bf16 D128 padded lastValid S6", H=10,
                seqlens_q=(520, 300, 130), seqlens_k=(1500, 3000, 200), d_qk=128, d_v=128,
                dtype="bf16", seed=43, n_per_block=128, split_kv=6, last_valid_kv_index=2000,
                seqused_k=(1400, 2500, 0)),
    wl.Workload("persist causal bf16 D128 split 1", H=16, seqlens_q=(513, 300, 260, 400),
                seqlens_k=(1000, 800, 1500, 2000), d_qk=128, d_v=128, dtype="bf16", seed=44,
                n_per_block=128, split_kv=1, mask=wl.MASK_CAUSAL),
    wl.Workload("persist prefix -100 f16 D128 S4", H=16, seqlens_q=(1024,), seqlens_k=(1024,),
                d_qk=128, d_v=128, dtype="f16", seed=45, n_per_block=64, split_kv=4,
                mask=wl.MASK_PREFIX_CAUSAL, prefix_offset=-100),
]


@pytest.mark.parametrize("w", PERSIST, ids=lambda w: w.name)
def test_persistent_form_matches_oracle(w):
    (q, k, v), (qd, kd, vd) = _inputs(w)
    S = w.split_kv
    p = skv.params_for(w, DEV)
    assert skv.sk_partial_kernel_name(p, qd, kd, vd) == "partial_tc_persist"
    o_part, l_part, _ = H.run_partials(w, qd, kd, vd, DEV, S)
    ref_po, ref_pl = oracle.partials(H.oracle_problem(w, S), q, k, v)
    got_o = o_part.permute(2, 0, 1, 3).cpu().numpy()
    got_l = l_part.permute(2, 0, 1).cpu().numpy()
    H.assert_close(got_o, got_l, ref_po, ref_pl, w.dtype, "persistent partials")
    empty = np.isneginf(ref_pl)
    assert (got_o[empty] == 0).all() and np.isneginf(got_l[empty]).all()
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    out, lse, _ = H.run_fwd(w, qd, kd, vd, DEV)
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, w.dtype, "persistent forward")
    out3, lse3 = _three_call(w, qd, kd, vd, S)
    H.assert_close(H.to_np(out3), H.lse_np(lse3), ref_o, ref_l, w.dtype, "persistent three calls")


def test_persistent_form_on_the_masked_workload_full_size():
    """The masked f16 workload (512 units of one to four key tiles) runs on the persistent
    form; sampled rows of every mask variant against the oracle."""
    w = wl.MASKED_F16
    q, k, v = w.make_inputs(DEV)
    assert skv.sk_partial_kernel_name(skv.params_for(w, DEV), q, k, v) == "partial_tc_persist"
    for mask, po in ((wl.MASK_CAUSAL, 0), (wl.MASK_PREFIX_CAUSAL, 2048), (wl.MASK_PREFIX_CAUSAL, -256)):
        wm = w.with_(mask=mask, prefix_offset=po)
        rows = H.sample_rows(wm, head=64, tail=64, rand=64)
        ref_o, ref_l = oracle.attention(H.oracle_problem(wm, 1), q.cpu(), k.cpu(), v.cpu(), rows=rows)
        out, lse, _ = H.run_fwd(wm, q, k, v, DEV)
        H.assert_close(H.to_np(out, rows), H.lse_np(lse, rows), ref_o, ref_l, wm.dtype,
                       f"masked persistent po={po}")


@pytest.mark.parametrize("S,mask,heads,sq", [(8, wl.MASK_CAUSAL, 16, 300), (1, wl.MASK_NONE, 32, 600)])
def test_persistent_form_dense_layout_equals_varlen(S, mask, heads, sq):
    """[B, seq, H, D] tensors without cu_seqlens on the persistent form (partials and, at split 1,
    the output written directly) give the packed layout's results bit for bit."""
    w = wl.Workload("dense persistent", H=heads, seqlens_q=(sq, sq), seqlens_k=(1600, 1600),
                    d_qk=128, d_v=128, dtype="bf16", seed=46, n_per_block=128, split_kv=S,
                    mask=mask)
    (_, _, _), (qd, kd, vd) = _inputs(w)
    p = skv.params_for(w, DEV)
    assert skv.sk_partial_kernel_name(p, qd, kd, vd) == "partial_tc_persist"
    out, lse, _ = H.run_fwd(w, qd, kd, vd, DEV)
    p.cu_seqlens_q = p.cu_seqlens_k = None
    qb, kb, vb = (t.view(2, -1, heads, 128) for t in (qd, kd, vd))
    outb = torch.empty(2, sq, heads, 128, dtype=qd.dtype, device=DEV)
    lseb = torch.empty(heads, 2 * sq, dtype=torch.float32, device=DEV)
    ws = torch.empty(max(skv.sk_workspace_bytes(p), 1), dtype=torch.uint8, device=DEV)
    assert skv.sk_partial_kernel_name(p, qb, kb, vb) == "partial_tc_persist"
    skv.sk_attn_fwd(p, qb, kb, vb, outb, lseb, ws)
    torch.cuda.synchronize()
    assert torch.equal(outb.view_as(out), out) and torch.equal(lseb, lse)


@pytest.mark.parametrize("dtype,dqk,dv,mask,po,window", [
    ("bf16", 192, 128, wl.MASK_CAUSAL, 0, -1),
    ("f16", 128, 128, wl.MASK_PREFIX_CAUSAL, 300, 150),
    ("bf16", 64, 64, wl.MASK_NONE, 0, -1),
])
def test_cuda_core_kernel_for_other_m_blocks(dtype, dqk, dv, mask, po, window):
    """16-bit storage with an M block of 64 rows and more than 16 queries per sequence: neither
    tensor-core kernel nor the decode kernel applies, so the register-tiled CUDA-core kernel
    computes the partials (compared under the same partition) and the output."""
    w = _small(dtype, dqk, dv, mask=mask, po=po, S=3, bn=64, sq=(300, 1, 77, 200),
               sk=(1000, 5, 0, 513), window=window)
    (q, k, v), (qd, kd, vd) = _inputs(w)
    bm = 64
    p = skv.params_for(w, DEV, split_kv=3, block_m=bm)
    assert skv.sk_partial_kernel_name(p, qd, kd, vd) == "partial_fma"
    o_part = torch.empty(w.H, 3, w.total_q, w.d_v, dtype=torch.float32, device=DEV)
    l_part = torch.empty(w.H, 3, w.total_q, dtype=torch.float32, device=DEV)
    skv.sk_attn_partial_fwd(p, qd, kd, vd, o_part, l_part)
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=qd.dtype, device=DEV)
    lse = torch.empty(w.H, w.total_q, dtype=torch.float32, device=DEV)
    ws = torch.empty(max(skv.sk_workspace_bytes(p), 1), dtype=torch.uint8, device=DEV)
    skv.sk_attn_fwd(p, qd, kd, vd, out, lse, ws)
    torch.cuda.synchronize()
    ref_po, ref_pl = oracle.partials(H.oracle_problem(w, 3, block_m=bm), q, k, v)
    H.assert_close(o_part.permute(2, 0, 1, 3).cpu().numpy(), l_part.permute(2, 0, 1).cpu().numpy(),
                   ref_po, ref_pl, w.dtype, "partials")
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, w.dtype, "forward")


def _random_workload(seed: int) -> wl.Workload:
    """A seeded random small problem: 1-5 sequences of 0-700 queries and 0-1500 keys, every
    head-dim pair and storage type, any mask with a random offset, window, lastValid, padded
    key slots, key tile and split count."""
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 6))
    sq = tuple(int(x) for x in rng.integers(0, 701, B))
    if sum(sq) == 0:
        sq = (1,) + sq[1:]
    sk = tuple(int(x) for x in rng.integers(0, 1501, B))
    dqk, dv = [(64, 64), (128, 128), (192, 128)][int(rng.integers(0, 3))]
    dtype = ["bf16", "f16", "f32"][int(rng.integers(0, 3))]
    mask = int(rng.integers(0, 3))
    po = int(rng.integers(-300, 1500)) if mask == wl.MASK_PREFIX_CAUSAL else 0
    window = int(rng.integers(0, 800)) if mask != wl.MASK_NONE and rng.random() < 0.4 else -1
    lvi = int(rng.integers(0, 1500)) if rng.random() < 0.3 else -1
    used = tuple(int(min(x, y)) for x, y in zip(sk, rng.integers(0, 1600, B))) if rng.random() < 0.3 else None
    bn = int(rng.choice([16, 32, 64, 128, 256]))
    S = int(rng.choice([1, 2, 3, 4, 5, 8, 13, 32]))
    return wl.Workload(f"random {seed}", H=int(rng.integers(1, 5)), seqlens_q=sq, seqlens_k=sk,
                       d_qk=dqk, d_v=dv, dtype=dtype, seed=seed, n_per_block=bn, split_kv=S,
                       mask=mask, prefix_offset=po, last_valid_kv_index=lvi, window_left=window,
                       seqused_k=used)


@pytest.mark.parametrize("seed", range(32))
def test_random_problems_match_oracle(seed):
    """Seeded random problems through sk_attn_fwd (and its split counts) against the oracle."""
    w = _random_workload(seed)
    (q, k, v), (qd, kd, vd) = _inputs(w)
    if w.total_k == 0:   # K and V need a real buffer even when no sequence has a key
        kd = torch.zeros(1, w.H, w.d_qk, dtype=qd.dtype, device=DEV)
        vd = torch.zeros(1, w.H, w.d_v, dtype=qd.dtype, device=DEV)
    out, lse, p = H.run_fwd(w, qd, kd, vd, DEV)
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, w.dtype, w.name)
    counts = torch.empty(w.total_q, dtype=torch.int32, device=DEV)
    skv.sk_valid_split_counts(p, counts)
    assert np.array_equal(counts.cpu().numpy(), oracle.split_counts(H.oracle_problem(w, w.split_kv)))


def test_persistent_form_beyond_its_unit_table():
    """More than 16 rounds of units per CTA (40 sequences x 16 heads x 2 M blocks x split 4 =
    5120 units on 152 CTAs): the rounds past the CTA's table are looked up as they come.
    Sampled rows of every sequence against the oracle, and the partials of the last rows."""
    rng = np.random.default_rng(47)
    w = wl.Workload("persist many units", H=16,
                    seqlens_q=tuple(int(x) for x in rng.integers(257, 400, 40)),
                    seqlens_k=tuple(int(x) for x in rng.integers(300, 1200, 40)), d_qk=64, d_v=64,
                    dtype="bf16", seed=47, n_per_block=64, split_kv=4, mask=wl.MASK_CAUSAL)
    (q, k, v), (qd, kd, vd) = _inputs(w)
    p = skv.params_for(w, DEV)
    assert skv.sk_partial_kernel_name(p, qd, kd, vd) == "partial_tc_persist"
    rows = H.sample_rows(w, head=4, tail=4, rand=4)
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v, rows=rows)
    out, lse, _ = H.run_fwd(w, qd, kd, vd, DEV)
    H.assert_close(H.to_np(out, rows), H.lse_np(lse, rows), ref_o, ref_l, w.dtype, "many units")
    o_part, l_part, _ = H.run_partials(w, qd, kd, vd, DEV, 4)
    tail = rows[-64:]
    ref_po, ref_pl = oracle.partials(H.oracle_problem(w, 4), q, k, v, rows=tail)
    H.assert_close(o_part.permute(2, 0, 1, 3).cpu().numpy()[tail], l_part.permute(2, 0, 1).cpu().numpy()[tail],
                   ref_po, ref_pl, w.dtype, "many units partials")
