"""Host-side checks of the C ABI (no GPU): every declared symbol is exported,
argument validation returns the documented statuses before any launch, the
automatic split choice follows the pages' rule, and workspace sizes add up."""
from __future__ import annotations

import ctypes
import json
import os
import re

import pytest

import split_kv_attention_flash_gb300 as skv
from split_kv_attention_flash_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "splitkv.h")
FAKE = 0x7f0000001000          # a 4 KiB-aligned address that is never dereferenced

SK_OK, SK_ERR_INVALID_ARG, SK_ERR_UNSUPPORTED, SK_ERR_WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def L():
    _build.build()
    return skv.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sk_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary_calls():
    names = _declared_functions()
    for n in ("sk_valid_split_counts", "sk_attn_partial_fwd", "sk_combine", "sk_attn_fwd",
              "sk_workspace_bytes", "sk_auto_split_kv"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in _declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def _params(**kw):
    base = dict(B=2, H=4, max_seqlen_q=64, max_seqlen_k=512, total_q=100, total_k=700, d_qk=128,
                d_v=128, cu_seqlens_q=FAKE, cu_seqlens_k=FAKE + 256, n_per_block=64, split_kv=3)
    base.update(kw)
    return skv.Params(**base)


def _t(dtype=skv.SK_BF16, ptr=FAKE, sb=0, sr=512, sh=128):
    return skv._Tensor(ptr, dtype, sb, sr, sh)


def _fwd(L, p, q=None, k=None, v=None, out=None, ws=FAKE, ws_bytes=1 << 40):
    q, k, v, out = q or _t(), k or _t(), v or _t(), out or _t()
    return L.sk_attn_fwd(ctypes.byref(p.c()), q, k, v, out, None, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), SK_ERR_INVALID_ARG),
    (dict(H=0), SK_ERR_INVALID_ARG),
    (dict(total_q=-1), SK_ERR_INVALID_ARG),
    (dict(cu_seqlens_k=None), SK_ERR_INVALID_ARG),
    (dict(cu_seqlens_q=None, cu_seqlens_k=None), SK_ERR_INVALID_ARG),  # dense totals mismatch
    (dict(prefix_offset=3), SK_ERR_INVALID_ARG),
    (dict(mask=skv.MASK_CAUSAL, prefix_offset=3), SK_ERR_INVALID_ARG),
    (dict(mask=7), SK_ERR_INVALID_ARG),
    (dict(last_valid_kv_index=-2), SK_ERR_INVALID_ARG),
    (dict(n_per_block=0), SK_ERR_INVALID_ARG),
    (dict(split_kv=33), SK_ERR_INVALID_ARG),
    (dict(split_kv=-1), SK_ERR_INVALID_ARG),
    (dict(block_m=-4), SK_ERR_INVALID_ARG),
    (dict(softmax_scale=float("nan")), SK_ERR_INVALID_ARG),
    (dict(fuse_combine=2), SK_ERR_INVALID_ARG),
    (dict(window_left=-2), SK_ERR_INVALID_ARG),
    (dict(window_left=16), SK_ERR_INVALID_ARG),                 # a window needs a causal mask
    (dict(d_qk=96, d_v=96), SK_ERR_UNSUPPORTED),
    (dict(d_qk=128, d_v=64), SK_ERR_UNSUPPORTED),
])
def test_invalid_params_rejected_before_launch(L, kw, status):
    assert _fwd(L, _params(**kw)) == status


def test_invalid_tensors_rejected_before_launch(L):
    p = _params()
    assert _fwd(L, p, q=_t(ptr=0)) == SK_ERR_INVALID_ARG                   # null
    assert _fwd(L, p, q=_t(ptr=FAKE + 8)) == SK_ERR_UNSUPPORTED            # 8-byte aligned only
    assert _fwd(L, p, k=_t(sr=500 + 3)) == SK_ERR_UNSUPPORTED              # 1006-byte row stride
    assert _fwd(L, p, v=_t(dtype=skv.SK_F16)) == SK_ERR_UNSUPPORTED        # mixed storage types
    assert _fwd(L, p, out=_t(dtype=skv.SK_F32)) == SK_ERR_UNSUPPORTED      # output not storage type
    assert _fwd(L, p, q=_t(dtype=9)) == SK_ERR_INVALID_ARG
    assert _fwd(L, p, q=_t(sr=-512)) == SK_ERR_INVALID_ARG


def test_workspace_too_small(L):
    p = _params(split_kv=3)
    need = skv.sk_workspace_bytes(p)
    assert need > 0
    assert _fwd(L, p, ws_bytes=need - 1) == SK_ERR_WORKSPACE
    assert _fwd(L, p, ws=FAKE + 16, ws_bytes=need) == SK_ERR_INVALID_ARG  # not 256-byte aligned


def test_workspace_layout_sizes(L):
    def a256(x):
        return (x + 255) // 256 * 256
    for S, tq, H, dv in ((3, 100, 4, 128), (8, 16384, 12, 128), (2, 1, 1, 64)):
        p = _params(split_kv=S, total_q=tq, H=H, d_qk=dv, d_v=dv)
        tickets = p.B * H * ((p.max_seqlen_q + 255) // 256) * 4
        assert skv.sk_workspace_bytes(p) == (a256(4 * H * S * tq * dv) + a256(4 * H * S * tq)
                                            + a256(tickets))
    assert skv.sk_workspace_bytes(_params(split_kv=1)) == 0


def test_partial_and_combine_validation(L):
    p = _params()
    c = ctypes.byref(p.c())
    assert L.sk_attn_partial_fwd(c, _t(), _t(), _t(), None, FAKE, None) == SK_ERR_INVALID_ARG
    assert L.sk_attn_partial_fwd(c, _t(), _t(), _t(), FAKE + 4, FAKE, None) == SK_ERR_UNSUPPORTED
    assert L.sk_combine(c, FAKE, FAKE, None, _t(), None, None) == SK_ERR_INVALID_ARG
    assert L.sk_valid_split_counts(c, None, None) == SK_ERR_INVALID_ARG
    assert L.sk_valid_split_counts(None, FAKE, None) == SK_ERR_INVALID_ARG


def test_auto_split_boundary_from_the_pages(L):
    data = json.load(open(os.path.join(ROOT, "tests", "golden", "auto_split_boundary.json")))
    for c in data["cases"]:
        p = _params(B=1, H=c["H"], max_seqlen_q=c["max_seqlen_q"], max_seqlen_k=c["max_seqlen_k"],
                    total_q=c["max_seqlen_q"], total_k=c["max_seqlen_k"], split_kv=0,
                    block_m=data["block_m"])
        assert skv.sk_choose_split_kv(p, data["sm_count"]) == c["split_kv"], c


def test_auto_split_rules(L):
    # forced values pass through
    for s in range(1, 33):
        assert skv.sk_choose_split_kv(_params(split_kv=s), 152) == s
    # single-query problems: smallest S with B*H*S >= 2*SM
    dec = dict(max_seqlen_q=1, max_seqlen_k=100000, total_q=32, total_k=3200000, split_kv=0)
    assert skv.sk_choose_split_kv(_params(B=32, H=32, **dec), 152) == 1
    assert skv.sk_choose_split_kv(_params(B=4, H=8, **dec), 152) == 10
    assert skv.sk_choose_split_kv(_params(B=1, H=8, **dec), 152) == 32
    # the default M block enters Q_tiles
    p = _params(B=1, H=12, max_seqlen_q=4096, max_seqlen_k=42700, total_q=4096, total_k=42700,
                split_kv=0)
    assert skv.sk_default_block_m(192, 128) == 256
    assert skv.sk_choose_split_kv(p, 152) == 3


def test_auto_split_keeps_windowed_problems_unsplit_when_the_first_split_is_hidden(L):
    # the window workload: the last 4096 queries of 42700 keys, window 8192. Split 0 of 3
    # holds keys [0, 14336); the deepest row's window starts at 42699 - 8191 = 34508.
    base = dict(B=1, H=12, max_seqlen_q=4096, max_seqlen_k=42700, total_q=4096, total_k=42700,
                split_kv=0, mask=2, prefix_offset=42700 - 4096, d_qk=192, d_v=128, n_per_block=128)
    assert skv.sk_choose_split_kv(_params(**base), 152) == 3
    assert skv.sk_choose_split_kv(_params(**base, window_left=8191), 152) == 1
    # the boundary: the deepest window start equal to the first split's end hides it
    assert skv.sk_choose_split_kv(_params(**base, window_left=42699 - 14336), 152) == 1
    assert skv.sk_choose_split_kv(_params(**base, window_left=42699 - 14335), 152) == 3
    # a window wider than the context hides nothing
    assert skv.sk_choose_split_kv(_params(**base, window_left=50000), 152) == 3
    # lastValid shortens the partition: 20000 keys in tiles of 128 give a first split of
    # 128 * ceil(157 / 3) = 6784 keys; the window start 34508 is past it
    assert skv.sk_choose_split_kv(_params(**base, window_left=8191, last_valid_kv_index=19999),
                                  152) == 1
    # plain causal ignores prefix_offset; Sq = Sk = 16384, first split 5504 keys
    c = dict(B=1, H=4, max_seqlen_q=16384, max_seqlen_k=16384, total_q=16384, total_k=16384,
             split_kv=0, mask=1, n_per_block=128)
    assert skv.sk_choose_split_kv(_params(**c, window_left=16383 - 5504), 152) == 1
    assert skv.sk_choose_split_kv(_params(**c, window_left=16383 - 5503), 152) == 3
    # no mask: the window is not applied, nor is the rule
    assert skv.sk_choose_split_kv(_params(**dict(base, mask=0, prefix_offset=0), window_left=10),
                                  152) == 3
    # a forced split is returned unchanged
    assert skv.sk_choose_split_kv(_params(**dict(base, split_kv=4), window_left=8191), 152) == 4


def test_selftest_limit_is_checked_before_any_launch(L):
    fn = L.sk_selftest_bounded_wait
    fn.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]
    assert fn(3_000_000_000, None) == SK_ERR_INVALID_ARG


def test_status_strings(L):
    for code in range(6):
        assert skv.sk_status_string(code)
    assert "unknown" in skv.sk_status_string(99)
    assert L.sk_version() >= 100
    assert L.sk_supported_head_dims(192, 128) and not L.sk_supported_head_dims(192, 192)


def _host_fwd(L, p, q=None, k=None, v=None, out=None, buf=FAKE, nbytes=1 << 40):
    fn = L.sk_attn_fwd_host
    fn.argtypes = [ctypes.POINTER(skv._Params), skv._Tensor, skv._Tensor, skv._Tensor, skv._Tensor,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    q, k, v, out = q or _t(), k or _t(), v or _t(), out or _t()
    return fn(ctypes.byref(p.c()), q, k, v, out, None, buf, nbytes, None)


def test_host_entry_buffer_layout(L):
    def a256(x):
        return (x + 255) // 256 * 256
    p = _params(split_kv=3)
    ws = skv.sk_workspace_bytes(p)
    es = 2
    q, kk = p.total_q * p.H * p.d_qk * es, p.total_k * p.H * p.d_qk * es
    v, o, lse = p.total_k * p.H * p.d_v * es, p.total_q * p.H * p.d_v * es, p.H * p.total_q * 4
    assert skv.sk_host_buffer_bytes(p, skv.SK_BF16, True) == (a256(q) + a256(kk) + a256(v) + a256(o)
                                                              + a256(lse) + a256(ws))
    assert skv.sk_host_buffer_bytes(p, skv.SK_BF16, False) == (a256(q) + a256(kk) + a256(v) + a256(o)
                                                               + a256(ws))
    assert (skv.sk_host_buffer_bytes(p, skv.SK_F32, False) - a256(ws)
            == a256(2 * q) + a256(2 * kk) + a256(2 * v) + a256(2 * o))


def test_host_entry_rejected_before_any_copy(L):
    p = _params(split_kv=3)
    need = skv.sk_host_buffer_bytes(p, skv.SK_BF16, False)
    assert _host_fwd(L, p, q=_t(ptr=0)) == SK_ERR_INVALID_ARG                 # null host tensor
    assert _host_fwd(L, p, k=_t(sr=1024)) == SK_ERR_UNSUPPORTED               # rows not packed
    assert _host_fwd(L, p, v=_t(sh=256, sr=1024)) == SK_ERR_UNSUPPORTED       # heads not packed
    assert _host_fwd(L, p, out=_t(dtype=skv.SK_F16)) == SK_ERR_UNSUPPORTED    # mixed storage types
    assert _host_fwd(L, p, nbytes=need - 1) == SK_ERR_WORKSPACE
    assert _host_fwd(L, p, buf=FAKE + 16, nbytes=need) == SK_ERR_INVALID_ARG  # not 256-byte aligned
    assert _host_fwd(L, p, buf=0, nbytes=need) == SK_ERR_INVALID_ARG
    assert _host_fwd(L, _params(B=0)) == SK_ERR_INVALID_ARG
