"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself:
  * the per-row split counts worked out on "Recombine fully masked split-KV
    attention partials on the host" (review notes on the per-row mask test);
  * the review notes' conservativeness argument (the host count never drops a
    split that holds a row's keys under the kernel's block-last-row partition,
    is >= 1 and <= split_kv), by brute force over small shapes;
  * a library attention routine (torch scaled_dot_product_attention and
    logsumexp in double precision) with a mask built from the visibility rule;
  * closed forms (zero queries -> mean of the visible values, LSE = log count;
    a single visible key -> that key's value);
  * the merge identity: merging the partials equals unsplit attention, and the
    NaN-safe clamps of computeFinalAttentionStage;
  * exact widening of every bf16 and f16 bit pattern.
Each check is a plain function so that test_oracle_mutants.py can run them
against copies of oracle.c with planted mistakes.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
MASKS = {"none": orc.MASK_NONE, "causal": orc.MASK_CAUSAL, "prefix_causal": orc.MASK_PREFIX_CAUSAL}


# ----------------------------------------------------------------- helpers

def _visible_matrix(sq, sk, mask, po, lvi, window=-1, used=None):
    """Visibility straight from the page's wording: key j is valid when
    j <= lastValid (last_valid_kv_index, default seq_len_k - 1), and under a
    causal / prefix-causal mask also j <= q + prefix_offset; a sliding window keeps
    j >= q + offset - window; keys at or past `used` are padding."""
    n = sk if used is None else min(sk, max(used, 0))
    last = n - 1 if lvi < 0 else min(lvi, n - 1)
    q = np.arange(sq)[:, None]
    j = np.arange(sk)[None, :]
    vis = j <= last
    if mask != orc.MASK_NONE:
        off = po if mask == orc.MASK_PREFIX_CAUSAL else 0
        vis = vis & (j <= q + off)
        if window >= 0:
            vis = vis & (j >= q + off - window)
    return np.broadcast_to(vis, (sq, sk)).copy()


def _random_problem(rng, B, H, dqk, dv, mask, po=0, lvi=-1, bn=16, S=3, bm=16,
                    sq_max=24, sk_max=70, allow_empty=True, window=-1, padded=False):
    lo = 0 if allow_empty else 1
    sq = [int(rng.integers(1, sq_max + 1)) for _ in range(B)]
    sk = [int(rng.integers(lo, sk_max + 1)) for _ in range(B)]
    cu_q = np.concatenate([[0], np.cumsum(sq)]).tolist()
    cu_k = np.concatenate([[0], np.cumsum(sk)]).tolist()
    used = [int(rng.integers(0, n + 3)) for n in sk] if padded else None
    prob = orc.Problem(cu_q=cu_q, cu_k=cu_k, H=H, d_qk=dqk, d_v=dv, mask=mask, prefix_offset=po,
                       last_valid_kv_index=lvi, n_per_block=bn, split_kv=S, block_m=bm,
                       window_left=window, seqused_k=used)
    g = torch.Generator().manual_seed(int(rng.integers(1 << 30)))
    q = torch.randn(cu_q[-1], H, dqk, generator=g, dtype=torch.float64)
    k = torch.randn(cu_k[-1], H, dqk, generator=g, dtype=torch.float64)
    v = torch.randn(cu_k[-1], H, dv, generator=g, dtype=torch.float64)
    return prob, q, k, v


def _library_attention(prob, q, k, v, key_range=None):
    """torch SDPA + logsumexp in f64 per sequence; rows with no visible key get
    NaN from SDPA and are reported in the returned `empty` mask instead."""
    H, scale = prob.H, 1.0 / math.sqrt(prob.d_qk) if prob.scale is None else prob.scale
    outs, lses, empties = [], [], []
    for b in range(prob.B):
        q0, q1 = prob.cu_q[b], prob.cu_q[b + 1]
        k0, k1 = prob.cu_k[b], prob.cu_k[b + 1]
        sq, sk = q1 - q0, k1 - k0
        used = None if prob.seqused_k is None else prob.seqused_k[b]
        vis = _visible_matrix(sq, sk, prob.mask, prob.prefix_offset, prob.last_valid_kv_index,
                              prob.window_left, used)
        if key_range is not None:
            kb, ke = key_range(b)
            inr = np.zeros((sq, sk), dtype=bool)
            for r in range(sq):
                inr[r, kb[r]:ke[r]] = True
            vis = vis & inr
        empty = ~vis.any(axis=1)
        qb = q[q0:q1].transpose(0, 1)
        kb_ = k[k0:k1].transpose(0, 1)
        vb = v[k0:k1].transpose(0, 1)
        m = torch.from_numpy(vis)
        if sk == 0:
            o = torch.zeros(H, sq, prob.d_v, dtype=torch.float64)
            lse = torch.full((H, sq), -math.inf, dtype=torch.float64)
        else:
            o = torch.nn.functional.scaled_dot_product_attention(qb, kb_, vb, attn_mask=m,
                                                                 scale=scale)
            sc = torch.matmul(qb, kb_.transpose(1, 2)) * scale
            sc = sc.masked_fill(~m, -math.inf)
            lse = torch.logsumexp(sc, dim=-1)
        outs.append(o.transpose(0, 1).numpy())
        lses.append(lse.transpose(0, 1).numpy())
        empties.append(empty)
    return np.concatenate(outs), np.concatenate(lses), np.concatenate(empties)


def _compare_to_library(out, lse, ref_o, ref_l, empty, tol=1e-12):
    full = ~empty
    assert np.isfinite(out).all(), "oracle produced a non-finite output"
    assert np.abs(out[full] - ref_o[full]).max(initial=0) < tol
    assert np.abs(lse[full] - ref_l[full]).max(initial=0) < tol
    assert (out[empty] == 0).all(), "fully masked rows must give an exact zero row"
    assert np.isneginf(lse[empty]).all(), "fully masked rows must give LSE = -inf"


# ------------------------------------------------------------- check bodies

def check_worked_counts():
    data = json.load(open(os.path.join(GOLDEN, "split_counts_worked_examples.json")))
    for c in data["cases"]:
        expect = c.get("counts")
        if expect is None:
            expect = [v for n, v in c["counts_runs"] for _ in range(n)]
        for sk in (c["seq_len_k"], c["seq_len_k"] + 37, 4 * c["seq_len_k"] + 1):
            p = orc.Problem(cu_q=[0, c["seq_len_q"]], cu_k=[0, sk], H=1, d_qk=8, d_v=8,
                            mask=MASKS[c["mask"]], prefix_offset=c["prefix_offset"],
                            n_per_block=c["n_per_block"], split_kv=c["split_kv"])
            got = orc.split_counts(p).tolist()
            assert got == expect, (c["name"], sk, got)


def check_counts_bruteforce(n_configs=2500, seed=11):
    """Conservativeness of the counts against the kernel partition."""
    rng = np.random.default_rng(seed)
    for _ in range(n_configs):
        sq = int(rng.choice([1, 2, 5, 17, 33, 40]))
        sk = int(rng.choice([0, 1, 7, 32, 33, 63, 80]))
        bn = int(rng.choice([1, 3, 16, 32]))
        S = int(rng.integers(1, 7))
        bm = int(rng.choice([1, 7, 16, 32, 256]))
        mask = int(rng.integers(0, 3))
        po = int(rng.integers(-sq - 2, sk + 3)) if mask == orc.MASK_PREFIX_CAUSAL else 0
        lvi = int(rng.choice([-1, -1, 0, 20, 1000]))
        window = int(rng.choice([-1, -1, 0, 5, 40])) if mask != orc.MASK_NONE else -1
        used = int(rng.integers(0, sk + 2)) if rng.random() < 0.3 else None
        p = orc.Problem(cu_q=[0, sq], cu_k=[0, sk], H=1, d_qk=4, d_v=4, mask=mask,
                        prefix_offset=po, last_valid_kv_index=lvi, n_per_block=bn, split_kv=S,
                        block_m=bm, window_left=window,
                        seqused_k=None if used is None else [used])
        counts = orc.split_counts(p)
        kb, ke = orc.split_ranges(p)
        vis = _visible_matrix(sq, sk, mask, po, lvi, window, used)
        j = np.arange(sk)
        in_split = (j[None, None, :] >= kb[:, :, None]) & (j[None, None, :] < ke[:, :, None])
        holds = (in_split & vis[:, None, :]).any(axis=2)                 # [sq, S]
        # every visible key sits in exactly one split of its row's block
        assert ((in_split & vis[:, None, :]).sum(axis=1) == vis).all()
        # splits are ordered, contiguous and disjoint
        nonempty = ke > kb
        assert (kb[:, 1:][nonempty[:, 1:]] >= ke[:, :-1][nonempty[:, 1:]]).all()
        needed = np.where(holds.any(axis=1), S - np.argmax(holds[:, ::-1], axis=1), 1)
        assert (counts >= 1).all() and (counts <= S).all()
        assert (counts >= needed).all(), (sq, sk, bn, S, bm, mask, po, lvi)
        if bm == 1 and sk > 0 and (used is None or used > 0):
            # one row per block: the kernel's partition is the row's own, so the
            # count is exactly the number of non-empty splits
            assert (counts == nonempty.sum(axis=1)).all()


def check_attention_vs_library(seed=5):
    rng = np.random.default_rng(seed)
    cases = [(orc.MASK_NONE, 0, -1), (orc.MASK_CAUSAL, 0, -1), (orc.MASK_PREFIX_CAUSAL, 9, -1),
             (orc.MASK_PREFIX_CAUSAL, -6, 30), (orc.MASK_NONE, 0, 12)]
    for mask, po, lvi in cases:
        prob, q, k, v = _random_problem(rng, B=3, H=3, dqk=24, dv=16, mask=mask, po=po, lvi=lvi)
        out, lse = orc.attention(prob, q, k, v, nthreads=2)
        ref_o, ref_l, empty = _library_attention(prob, q, k, v)
        _compare_to_library(out, lse, ref_o, ref_l, empty)


def check_window_and_padding_vs_library(seed=12):
    """Sliding window ([P2]: the forced split honours the caller's window) and padded key
    slots with a per-sequence used count ([P2]: padded cu_seqlens): unsplit attention
    and every split's partial against the library routine, and merge == unsplit."""
    rng = np.random.default_rng(seed)
    for mask, po, window, padded in ((orc.MASK_CAUSAL, 0, 6, False),
                                     (orc.MASK_PREFIX_CAUSAL, 25, 17, True),
                                     (orc.MASK_PREFIX_CAUSAL, -4, 0, True),
                                     (orc.MASK_NONE, 0, -1, True)):
        prob, q, k, v = _random_problem(rng, B=3, H=2, dqk=16, dv=8, mask=mask, po=po, bn=8,
                                        S=4, bm=8, window=window, padded=padded)
        out, lse = orc.attention(prob, q, k, v, nthreads=2)
        ref_o, ref_l, empty = _library_attention(prob, q, k, v)
        _compare_to_library(out, lse, ref_o, ref_l, empty)
        o_part, l_part = orc.partials(prob, q, k, v)
        kb, ke = orc.split_ranges(prob)
        for s_ in range(prob.split_kv):
            def key_range(b, s_=s_):
                r0, r1 = prob.cu_q[b], prob.cu_q[b + 1]
                return kb[r0:r1, s_], ke[r0:r1, s_]
            r_o, r_l, emp = _library_attention(prob, q, k, v, key_range=key_range)
            _compare_to_library(o_part[:, :, s_], l_part[:, :, s_], r_o, r_l, emp)
        out_m, lse_m = orc.merge(o_part, l_part, orc.split_counts(prob))
        assert np.abs(out_m - out).max() < 1e-12
        fin = np.isfinite(lse)
        assert np.array_equal(np.isneginf(lse_m), ~fin)
        assert np.abs(lse_m[fin] - lse[fin]).max(initial=0) < 1e-12


def check_attention_closed_forms(seed=6):
    rng = np.random.default_rng(seed)
    # zero queries: every visible score is 0
    prob, q, k, v = _random_problem(rng, B=2, H=2, dqk=8, dv=8, mask=orc.MASK_PREFIX_CAUSAL,
                                    po=3, allow_empty=False)
    q.zero_()
    out, lse = orc.attention(prob, q, k, v)
    for b in range(prob.B):
        sq = prob.cu_q[b + 1] - prob.cu_q[b]
        sk = prob.cu_k[b + 1] - prob.cu_k[b]
        vis = _visible_matrix(sq, sk, prob.mask, 3, -1)
        vb = v[prob.cu_k[b]:prob.cu_k[b + 1]].numpy()
        for r in range(sq):
            n = vis[r].sum()
            row = prob.cu_q[b] + r
            if n == 0:
                assert (out[row] == 0).all() and np.isneginf(lse[row]).all()
                continue
            assert np.allclose(out[row], vb[vis[r]].mean(axis=0), atol=1e-13, rtol=0)
            assert np.allclose(lse[row], math.log(n), atol=1e-13, rtol=0)
    # one visible key: row 0 of a causal sequence sees key 0 only
    prob, q, k, v = _random_problem(rng, B=2, H=3, dqk=8, dv=5, mask=orc.MASK_CAUSAL,
                                    allow_empty=False)
    out, lse = orc.attention(prob, q, k, v)
    for b in range(prob.B):
        r0, k0 = prob.cu_q[b], prob.cu_k[b]
        assert np.array_equal(out[r0], v[k0].numpy())
        s = (q[r0] * k[k0]).sum(-1).numpy() / math.sqrt(prob.d_qk)
        assert np.allclose(lse[r0], s, atol=1e-13, rtol=0)


def check_partials_vs_library(seed=7):
    rng = np.random.default_rng(seed)
    for mask, po in ((orc.MASK_NONE, 0), (orc.MASK_CAUSAL, 0), (orc.MASK_PREFIX_CAUSAL, 11)):
        prob, q, k, v = _random_problem(rng, B=2, H=2, dqk=16, dv=8, mask=mask, po=po, bn=8,
                                        S=4, bm=8)
        o_part, l_part = orc.partials(prob, q, k, v)
        kb, ke = orc.split_ranges(prob)
        for s in range(prob.split_kv):
            def key_range(b, s=s):
                r0, r1 = prob.cu_q[b], prob.cu_q[b + 1]
                return kb[r0:r1, s], ke[r0:r1, s]
            ref_o, ref_l, empty = _library_attention(prob, q, k, v, key_range=key_range)
            _compare_to_library(o_part[:, :, s], l_part[:, :, s], ref_o, ref_l, empty)


def check_merge_equals_unsplit(seed=8):
    rng = np.random.default_rng(seed)
    for mask, po, lvi, S, bm in ((orc.MASK_NONE, 0, -1, 3, 16), (orc.MASK_CAUSAL, 0, -1, 4, 8),
                                 (orc.MASK_PREFIX_CAUSAL, 20, 40, 5, 16),
                                 (orc.MASK_PREFIX_CAUSAL, -5, -1, 2, 4),
                                 (orc.MASK_CAUSAL, 0, -1, 6, 1)):
        prob, q, k, v = _random_problem(rng, B=3, H=2, dqk=12, dv=10, mask=mask, po=po, lvi=lvi,
                                        bn=8, S=S, bm=bm)
        o_part, l_part = orc.partials(prob, q, k, v)
        counts = orc.split_counts(prob)
        out_m, lse_m = orc.merge(o_part, l_part, counts)
        out, lse = orc.attention(prob, q, k, v)
        assert np.isfinite(out_m).all()
        assert np.abs(out_m - out).max() < 1e-12
        fin = np.isfinite(lse)
        assert np.array_equal(np.isneginf(lse_m), ~fin)
        assert np.abs(lse_m[fin] - lse[fin]).max(initial=0) < 1e-12


def check_merge_clamps(seed=9):
    rng = np.random.default_rng(seed)
    n, H, S, dv = 6, 2, 5, 7
    o = rng.standard_normal((n, H, S, dv))
    # every valid split empty: weights are exactly 0, output row is exactly 0
    l_all = np.full((n, H, S), -np.inf)
    out, lse = orc.merge(o, l_all, np.full(n, S, np.int32))
    assert (out == 0).all() and np.isneginf(lse).all()
    # splits s >= count are never read: poison them with NaN
    l = rng.standard_normal((n, H, S)) * 3
    counts = np.array([1, 2, 3, 5, 4, 2], np.int32)
    o_p, l_p = o.copy(), l.copy()
    for i, c in enumerate(counts):
        o_p[i, :, c:] = np.nan
        l_p[i, :, c:] = np.nan
    out, lse = orc.merge(o_p, l_p, counts)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    for i, c in enumerate(counts):
        ref_l = np.logaddexp.reduce(l[i, :, :c], axis=-1)
        ref_o = (np.exp(l[i, :, :c] - ref_l[:, None])[..., None] * o[i, :, :c]).sum(axis=1)
        assert np.abs(lse[i] - ref_l).max() < 1e-13
        assert np.abs(out[i] - ref_o).max() < 1e-13
    # a single valid split is passed through unchanged
    out, lse = orc.merge(o, l, np.ones(n, np.int32))
    assert np.array_equal(out, o[:, :, 0]) and np.array_equal(lse, l[:, :, 0])
    # mixed: one finite split among -inf ones
    l_mix = np.full((n, H, S), -np.inf)
    l_mix[:, :, 2] = 0.25
    out, lse = orc.merge(o, l_mix, np.full(n, S, np.int32))
    assert np.array_equal(out, o[:, :, 2]) and np.array_equal(lse, l_mix[:, :, 2])


def check_split_one_is_unsplit(seed=10):
    rng = np.random.default_rng(seed)
    prob, q, k, v = _random_problem(rng, B=2, H=2, dqk=8, dv=8, mask=orc.MASK_CAUSAL, S=1)
    o_part, l_part = orc.partials(prob, q, k, v)
    out, lse = orc.attention(prob, q, k, v)
    out_m, lse_m = orc.merge(o_part, l_part, orc.split_counts(prob))
    assert np.array_equal(o_part[:, :, 0], out) and np.array_equal(l_part[:, :, 0], lse)
    assert np.array_equal(out_m, out) and np.array_equal(lse_m, lse)


def check_storage_widening():
    """Every bf16 / f16 bit pattern widens exactly: with one query and one key
    per sequence the output is that key's value."""
    n = 1 << 16
    bits = torch.arange(n, dtype=torch.int32).to(torch.int16)
    for dt, ref in ((torch.bfloat16, bits.view(torch.bfloat16).double()),
                    (torch.float16, torch.from_numpy(bits.numpy().view(np.float16).astype(np.float64)))):
        cu = list(range(n + 1))
        prob = orc.Problem(cu_q=cu, cu_k=cu, H=1, d_qk=1, d_v=1)
        q = torch.zeros(n, 1, 1, dtype=dt)
        v = bits.view(dt).reshape(n, 1, 1)
        out, _ = orc.attention(prob, q, q, v)
        got = torch.from_numpy(out[:, 0, 0])
        assert torch.equal(torch.isnan(got), torch.isnan(ref))
        fin = ~torch.isnan(ref)
        assert torch.equal(got[fin], ref[fin])


ALL_CHECKS = [check_worked_counts, check_counts_bruteforce, check_attention_vs_library,
              check_window_and_padding_vs_library,
              check_attention_closed_forms, check_partials_vs_library, check_merge_equals_unsplit,
              check_merge_clamps, check_split_one_is_unsplit, check_storage_widening]


# ------------------------------------------------------------------- tests

@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        orc.split_counts(orc.Problem(cu_q=[0, 4], cu_k=[0, 8], H=1, d_qk=4, d_v=4, n_per_block=0))
    with pytest.raises(ValueError):
        orc.split_counts(orc.Problem(cu_q=[0, 4], cu_k=[0, 8], H=1, d_qk=4, d_v=4, split_kv=0))
    with pytest.raises(ValueError):
        orc.split_counts(orc.Problem(cu_q=[0, 4], cu_k=[0, 8], H=1, d_qk=4, d_v=4,
                                     last_valid_kv_index=-2))
    with pytest.raises(ValueError):   # a window needs a causal mask
        orc.split_counts(orc.Problem(cu_q=[0, 4], cu_k=[0, 8], H=1, d_qk=4, d_v=4, window_left=3))
