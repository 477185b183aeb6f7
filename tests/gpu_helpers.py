"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same stored inputs, compare with the stated tolerances.

Tolerances (split counts bit-exact; outputs against the f64 oracle):
  f32 storage       O max-abs <= 1e-5
  bf16/f16 storage  O max-abs <= 2e-2 and cosine similarity >= 0.9999
  LSE               max-abs <= 1e-4 on finite entries; -inf exactly where expected
  no NaN anywhere; fully masked rows are an exact 0 row.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import split_kv_attention_flash_gb300 as skv

TOL_O = {"f32": 1e-5, "bf16": 2e-2, "f16": 2e-2}
TOL_LSE = 1e-4
MIN_COS = 0.9999


def oracle_problem(w, S: int, block_m: int | None = None) -> oracle.Problem:
    return oracle.Problem(cu_q=w.cu_seqlens_q, cu_k=w.cu_seqlens_k, H=w.H, d_qk=w.d_qk,
                          d_v=w.d_v, mask=w.mask, prefix_offset=w.prefix_offset,
                          last_valid_kv_index=w.last_valid_kv_index, n_per_block=w.n_per_block,
                          split_kv=S, block_m=block_m or skv.sk_default_block_m(w.d_qk, w.d_v),
                          window_left=w.window_left,
                          seqused_k=None if w.seqused_k is None else list(w.seqused_k))


def resolved_split(w, dev) -> int:
    return skv.sk_auto_split_kv(skv.params_for(w, dev))


def run_fwd(w, qd, kd, vd, dev, split_kv=None, with_lse=True, fuse_combine=0):
    p = skv.params_for(w, dev, split_kv=split_kv, fuse_combine=fuse_combine)
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=qd.dtype, device=dev)
    lse = torch.empty(w.H, w.total_q, dtype=torch.float32, device=dev) if with_lse else None
    nbytes = skv.sk_workspace_bytes(p)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
    skv.sk_attn_fwd(p, qd, kd, vd, out, lse, ws)
    torch.cuda.synchronize()
    return out, lse, p


def run_partials(w, qd, kd, vd, dev, S):
    p = skv.params_for(w, dev, split_kv=S)
    o_part = torch.empty(w.H, S, w.total_q, w.d_v, dtype=torch.float32, device=dev)
    l_part = torch.empty(w.H, S, w.total_q, dtype=torch.float32, device=dev)
    skv.sk_attn_partial_fwd(p, qd, kd, vd, o_part, l_part)
    torch.cuda.synchronize()
    return o_part, l_part, p


def sample_rows(w, head=64, tail=64, rand=64, seed=0) -> np.ndarray:
    """Per sequence: the first `head`, last `tail` and `rand` seeded random rows."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(w.B):
        q0, q1 = w.cu_seqlens_q[b], w.cu_seqlens_q[b + 1]
        n = q1 - q0
        sel = set(range(q0, q0 + min(head, n))) | set(range(max(q0, q1 - tail), q1))
        if n > 0:
            sel |= set(int(x) for x in rng.integers(q0, q1, size=min(rand, n)))
        rows.extend(sorted(sel))
    return np.asarray(rows, dtype=np.int32)


def to_np(out: torch.Tensor, rows=None) -> np.ndarray:
    o = out.float().cpu().numpy()
    return o if rows is None else o[rows]


def lse_np(lse: torch.Tensor, rows=None) -> np.ndarray:
    l = lse.cpu().numpy().T          # [total_q, H]
    return l if rows is None else l[rows]


def assert_close(got_o, got_l, ref_o, ref_l, dtype: str, what: str = ""):
    got_o = np.asarray(got_o, dtype=np.float64)
    assert not np.isnan(got_o).any(), f"{what}: NaN in output"
    assert np.isfinite(got_o).all(), f"{what}: non-finite output"
    err = np.abs(got_o - ref_o).max(initial=0.0)
    assert err <= TOL_O[dtype], f"{what}: output max abs error {err:.3g} > {TOL_O[dtype]}"
    if dtype != "f32":
        a, b = got_o.ravel(), ref_o.ravel()
        na, nb = np.linalg.norm(a), np.linalg.norm(b)
        if nb > 0:
            cos = float(a @ b / (na * nb))
            assert cos >= MIN_COS, f"{what}: cosine {cos:.7f} < {MIN_COS}"
    if got_l is not None:
        got_l = np.asarray(got_l, dtype=np.float64)
        assert not np.isnan(got_l).any(), f"{what}: NaN in LSE"
        ref_inf = np.isneginf(ref_l)
        assert np.array_equal(np.isneginf(got_l), ref_inf), f"{what}: -inf LSE pattern differs"
        assert np.isfinite(got_l[~ref_inf]).all()
        lerr = np.abs(got_l[~ref_inf] - ref_l[~ref_inf]).max(initial=0.0)
        assert lerr <= TOL_LSE, f"{what}: LSE max abs error {lerr:.3g} > {TOL_LSE}"
        # a fully masked row is an exact zero row
        empty = np.broadcast_to(ref_inf[..., None], got_o.shape)
        assert (got_o[empty] == 0).all(), f"{what}: fully masked rows are not exactly 0"
