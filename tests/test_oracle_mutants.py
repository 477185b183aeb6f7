"""Plant plausible mistakes in copies of oracle.c and check that the pins catch
each one (no GPU). The committed oracle is never modified: every mutant is a
patched copy compiled into a temporary directory and exercised in a child
process, so that a mutant that crashes cannot take the test session down."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

import oracle as orc
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(orc.__file__), "oracle.c")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("count without the outer ceil", "c = ceil_div(n, keys_per_split);", "c = n / keys_per_split;"),
    ("count splits tiles by floor plus one", "ceil_div(ceil_div(n, p->n_per_block), p->split_kv)",
     "(ceil_div(n, p->n_per_block) / p->split_kv + 1)"),
    ("partition floors itersPerBlock", "long long iters = ceil_div(n_tiles, p->split_kv);",
     "long long iters = n_tiles / p->split_kv + (n_tiles < p->split_kv);"),
    ("partition uses the block's first row",
     "long long block_last = covered_last(p, b, last_row);",
     "long long block_last = covered_last(p, b, first_row);"),
    ("causal comparison off by one", "if ((long long)j > diag)", "if ((long long)j >= diag)"),
    ("prefix offset dropped", "return p->mask == ORC_MASK_PREFIX_CAUSAL ? p->prefix_offset : 0;",
     "return 0;"),
    ("last_valid_kv_index ignored", "if (p->last_valid_kv_index >= 0 && p->last_valid_kv_index < last)",
     "if (0)"),
    ("softmax scale dropped", "double sc = p->scale * dot;", "double sc = dot;"),
    ("sliding window ignored", "if (p->window_left >= 0 && (long long)j < diag - p->window_left)",
     "if (0)"),
    ("sliding window off by one", "(long long)j < diag - p->window_left)",
     "(long long)j <= diag - p->window_left)"),
    ("padded key slots used in full", "if (p->seqused_k && p->seqused_k[b] < n)", "if (0)"),
    ("key read with the wrong head", "orc_load(K, (krow * H + h) * dqk + d)",
     "orc_load(K, (krow * H + 0) * dqk + d)"),
    ("keys summed in place of values", "o[d] += w * orc_load(V, (krow * H + h) * dv + d);",
     "o[d] += w * orc_load(K, (krow * H + h) * dqk + d);"),
    ("query row taken from the key offsets", "const int64_t qrow = (int64_t)p->cu_q[b] + q;",
     "const int64_t qrow = (int64_t)p->cu_k[b] + q < (int64_t)p->cu_q[p->B] ? (int64_t)p->cu_k[b] + q : q;"),
    ("LSE without the max", "*lse = m + log(z);", "*lse = log(z);"),
    ("merge weight sign flipped", "double w = exp(l_part[slot0 + s] - m);",
     "double w = exp(m - l_part[slot0 + s]);"),
    ("merge without the weight-sum clamp", "double denom = wsum > 1.0 ? wsum : 1.0;",
     "double denom = wsum;"),
    ("merge without the max clamp", "double m = -DBL_MAX;", "double m = -INFINITY;"),
    ("merge reads every split", "for (int s = 0; s < count; ++s) {\n                double w",
     "for (int s = 0; s < S; ++s) {\n                double w"),
    ("f16 exponent bias off by one", "x = ldexp((double)(m + 1024), e - 25);",
     "x = ldexp((double)(m + 1024), e - 24);"),
]


def _build_mutant(tmpdir, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not unique or missing: {old!r}"
    src = os.path.join(tmpdir, "oracle.c")
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    hdr = os.path.join(os.path.dirname(SRC), "oracle.h")
    with open(os.path.join(tmpdir, "oracle.h"), "w") as f:
        f.write(open(hdr).read())
    so = os.path.join(tmpdir, "liboracle_mutant.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", src, "-o", so, "-lm"],
                   check=True)
    return so


def _run_checks(so: str) -> list:
    """Run every pin against the library at `so`; return the pins that failed."""
    orc.use_library(so)
    caught = []
    try:
        for check in pins.ALL_CHECKS:
            try:
                if check is pins.check_counts_bruteforce:
                    check(n_configs=600)
                else:
                    check()
            except (AssertionError, ValueError) as e:  # a pin failed: the mistake is caught
                caught.append(f"{check.__name__}: {str(e)[:60]}")
    finally:
        orc.use_library(None)
    return caught


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    so = _build_mutant(str(tmp_path), old, new)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "tests.test_oracle_mutants", so], cwd=root,
                       capture_output=True, text=True, timeout=600)
    # exit 0: at least one pin failed; 1: none did; anything else: the child crashed
    assert r.returncode != 1, f"no pin caught the planted mistake: {name}\n{r.stdout}{r.stderr}"
    assert r.returncode == 0, f"mutant crashed instead of failing a pin: {r.stderr[-2000:]}"


if __name__ == "__main__":
    failed = _run_checks(sys.argv[1])
    print("\n".join(failed))
    sys.exit(0 if failed else 1)
