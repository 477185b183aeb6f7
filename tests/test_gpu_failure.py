"""Failure detection on the GPU without a fault: every wait in the library's kernels is
bounded; when one runs out the kernel records a code in the library's device error word
and returns, and the host reads it as SK_ERR_TIMEOUT. The self-test kernel waits on a
barrier that nothing arrives on, so its wait must run out."""
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


def test_bounded_wait_runs_out_and_is_reported():
    torch.cuda.set_device(DEV)
    assert skv.sk_read_device_error(clear=True) == 0
    skv.sk_selftest_bounded_wait(20_000_000)               # 20 ms
    assert skv.sk_read_device_error(clear=True) == 0x401   # recorded, then cleared
    assert skv.sk_read_device_error(clear=True) == 0


def test_context_usable_after_a_timeout():
    skv.sk_selftest_bounded_wait(5_000_000)
    assert skv.sk_read_device_error(clear=True) == 0x401
    w = wl.Workload("after timeout", H=2, seqlens_q=(300,), seqlens_k=(900,), d_qk=128, d_v=128,
                    dtype="bf16", seed=31, n_per_block=128, split_kv=3, mask=wl.MASK_CAUSAL)
    q, k, v = w.make_inputs("cpu")
    out, lse, _ = H.run_fwd(w, q.to(DEV), k.to(DEV), v.to(DEV), DEV)
    ref_o, ref_l = oracle.attention(H.oracle_problem(w, 1), q, k, v)
    H.assert_close(H.to_np(out), H.lse_np(lse), ref_o, ref_l, "bf16", "after timeout")
    assert skv.sk_read_device_error(clear=True) == 0
