"""Seeded synthetic workloads for split-KV attention forward.

This module only describes shapes and draws random inputs. It holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Shapes follow the workloads on the pages:
  * "[ASM] [HIP] [JIT] [gfx942] Optimize long-context FMHA with split-KV",
    Motivation and Test Result: packed-varlen prefill, bf16, D_QK 192, D_V 128,
    12 heads, 4096 queries per sequence, 8K-128K keys; target shape Sq 4096,
    Sk 42700, H 12.
  * "Recombine fully masked split-KV attention partials on the host", Technical
    details and review notes: causal / prefix-causal masks, seq_len_q larger than
    the key tile, last_valid_kv_index.
No dataset or trained weights are involved: every value is drawn from a seeded
normal distribution and cast to the storage type.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

MASK_NONE, MASK_CAUSAL, MASK_PREFIX_CAUSAL = 0, 1, 2

_TORCH_DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    seqlens_q: tuple
    seqlens_k: tuple
    d_qk: int
    d_v: int
    dtype: str                      # "bf16" | "f16" | "f32"
    seed: int
    n_per_block: int = 128
    split_kv: int = 0               # 0: automatic choice
    mask: int = MASK_NONE
    prefix_offset: int = 0
    last_valid_kv_index: int = -1
    value_scale: float = 1.0        # inputs are N(0, 1) * value_scale
    window_left: int = -1           # sliding window (causal masks only), -1: none
    seqused_k: tuple | None = None  # keys used per sequence when key slots are padded
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def B(self) -> int:
        return len(self.seqlens_q)

    @property
    def cu_seqlens_q(self) -> list:
        return _cumsum(self.seqlens_q)

    @property
    def cu_seqlens_k(self) -> list:
        return _cumsum(self.seqlens_k)

    @property
    def total_q(self) -> int:
        return sum(self.seqlens_q)

    @property
    def total_k(self) -> int:
        return sum(self.seqlens_k)

    @property
    def max_seqlen_q(self) -> int:
        return max(self.seqlens_q) if self.seqlens_q else 0

    @property
    def max_seqlen_k(self) -> int:
        return max(self.seqlens_k) if self.seqlens_k else 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPES[self.dtype]

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    def make_inputs(self, device="cpu"):
        """Q [total_q, H, d_qk], K [total_k, H, d_qk], V [total_k, H, d_v] in the
        storage dtype, drawn in that order from one generator seeded with `seed`
        on `device`. The same seed on another device gives other values, so a
        test draws once and copies."""
        dev = torch.device(device)
        g = torch.Generator(device=dev)
        g.manual_seed(self.seed)
        out = []
        for rows, d in ((self.total_q, self.d_qk), (self.total_k, self.d_qk),
                        (self.total_k, self.d_v)):
            x = torch.randn((rows, self.H, d), generator=g, device=dev, dtype=torch.float32)
            if self.value_scale != 1.0:
                x.mul_(self.value_scale)
            out.append(x.to(self.torch_dtype))
        return tuple(out)


def _cumsum(lens) -> list:
    acc, out = 0, [0]
    for n in lens:
        acc += int(n)
        out.append(acc)
    return out


def decode_lengths(batch: int, lo: int, hi: int, seed: int) -> tuple:
    """Per-sequence key counts uniform on [lo, hi], drawn on the CPU."""
    g = torch.Generator()
    g.manual_seed(seed)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (batch,), generator=g))


# --- the workloads of the method's own statement, plus the target shape ------

TINY_CAUSAL = Workload("tiny causal f32 (B1 H2 Sq64 Sk256 D64, BN32, S4)", H=2,
                       seqlens_q=(64,), seqlens_k=(256,), d_qk=64, d_v=64, dtype="f32",
                       seed=0, n_per_block=32, split_kv=4, mask=MASK_CAUSAL)

NONCAUSAL_BF16 = Workload("non-causal bf16 (B2 H8 Sq512 Sk8192 D128, BN128)", H=8,
                          seqlens_q=(512, 512), seqlens_k=(8192, 8192), d_qk=128, d_v=128,
                          dtype="bf16", seed=1, n_per_block=128, split_kv=4)

MASKED_F16 = Workload("masked f16 (B1 H16 Sq2048 Sk4096 D128, BN64, S4, lastValid 3000)",
                      H=16, seqlens_q=(2048,), seqlens_k=(4096,), d_qk=128, d_v=128,
                      dtype="f16", seed=2, n_per_block=64, split_kv=4, mask=MASK_CAUSAL,
                      last_valid_kv_index=3000)

LONG_VARLEN = Workload("long-context varlen prefill bf16 (4 x Sq4096, Sk 8192/42700/65536/131072,"
                       " H12, D192/128)", H=12, seqlens_q=(4096,) * 4,
                       seqlens_k=(8192, 42700, 65536, 131072), d_qk=192, d_v=128, dtype="bf16",
                       seed=3, n_per_block=128, split_kv=0, value_scale=0.5)

TARGET_SHAPE = Workload("varlen prefill bf16 Sq4096 Sk42700 H12 D192/128 non-causal", H=12,
                        seqlens_q=(4096,), seqlens_k=(42700,), d_qk=192, d_v=128, dtype="bf16",
                        seed=3, n_per_block=128, split_kv=0, value_scale=0.5)

DECODE = Workload("decode bf16 (B32 H32 Sq1, Sk ~ U[4096, 131072], D128)", H=32,
                  seqlens_q=(1,) * 32, seqlens_k=decode_lengths(32, 4096, 131072, 4),
                  d_qk=128, d_v=128, dtype="bf16", seed=4, n_per_block=128, split_kv=0)

# the target shape with D_QK = D_V = 128, for comparing the head-dim configurations
TARGET_D128 = TARGET_SHAPE.with_(name="varlen prefill bf16 Sq4096 Sk42700 H12 D128/128 non-causal",
                                 d_qk=128, d_v=128)

# sliding-window prefill: the last 4096 queries of a 42700-key context, each seeing the
# 8192 keys up to its own position
WINDOW = TARGET_SHAPE.with_(name="sliding-window prefill bf16 Sq4096 Sk42700 H12 D192/128 window 8192",
                            mask=MASK_PREFIX_CAUSAL, prefix_offset=42700 - 4096, window_left=8191)

# multi-token decode: eight queries per sequence (speculative or batched decoding)
DECODE_MQ = DECODE.with_(name="multi-query decode bf16 (B32 H32 Sq8, Sk ~ U[4096, 131072], D128)",
                         seqlens_q=(8,) * 32)

# the masked workload under its prefix-causal mask: queries are the last 2048 positions of
# the 4096 keys (prefix_offset = Sk - Sq), so rows past 952 reach the last valid key 3000 and
# the splits beyond it hold no visible key
MASKED_PREFIX_F16 = MASKED_F16.with_(
    name="masked f16 prefix-causal (B1 H16 Sq2048 Sk4096 D128, offset 2048, BN64, S4, lastValid 3000)",
    mask=MASK_PREFIX_CAUSAL, prefix_offset=2048)

# causal self-attention prefill (not one of the pages' workloads: the usual causal shape,
# where later query blocks see more keys)
CAUSAL_PREFILL = Workload("causal prefill bf16 (B1 H16 Sq=Sk=16384, D128)", H=16, seqlens_q=(16384,),
                          seqlens_k=(16384,), d_qk=128, d_v=128, dtype="bf16", seed=5,
                          n_per_block=128, split_kv=0, mask=MASK_CAUSAL)

# a 4.3 GB decode case with the decode workload's layout (for profiler captures)
DECODE_SMALL = DECODE.with_(name="decode bf16 (B32 H32 Sq1, Sk 8192, D128)", seqlens_k=(8192,) * 32)

ALL = {"decode_small": DECODE_SMALL, "decode_mq": DECODE_MQ, "window": WINDOW, "tiny": TINY_CAUSAL, "noncausal": NONCAUSAL_BF16, "masked": MASKED_F16,
       "masked_prefix": MASKED_PREFIX_F16, "causal_prefill": CAUSAL_PREFILL,
       "varlen": LONG_VARLEN, "target": TARGET_SHAPE, "decode": DECODE, "target_d128": TARGET_D128}
