"""The benchmark's algorithmic counts (the numerators of every roofline
fraction) against brute-force enumeration: visible (query, key) pairs by the
visibility rule key j visible to the query at pos iff j <= pos and, with a
window W > 0, pos - j < W; the KV tokens any query of a sequence sees, each
counted once; the pages those tokens sit on.  Also the sliding-window
prefill's pair count that follows from "Chasing speed of light on TPU v6e"
(section "Attention": a key is seen by the W queries that follow it)."""

from __future__ import annotations

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from ragged_paged_attention_rpa_gb300 import workloads  # noqa: E402


def brute(b, part=None):
    pairs, tokens, pages = 0, 0, 0
    nq = 0
    for s in range(b.num_seqs):
        ql = int(b.cu_q_lens[s + 1] - b.cu_q_lens[s])
        if ql == 0 or (part == "decode" and ql != 1) or (part == "prefill" and ql == 1):
            continue
        nq += ql
        L = int(b.kv_lens[s])
        W = 0 if b.window is None else int(b.window[s])
        seen = set()
        for i in range(ql):
            pos = L - ql + i
            for j in range(L):
                if j <= pos and (W <= 0 or pos - j < W):
                    pairs += 1
                    seen.add(j)
        tokens += len(seen)
        pages += len({j // b.page_size for j in seen})
    return pairs, tokens, pages, nq


@pytest.mark.parametrize("seed", range(6))
def test_counts_match_brute_force(seed):
    rng = np.random.default_rng(600 + seed)
    n = int(rng.integers(1, 9))
    ql = rng.integers(1, 40, size=n)
    kv = (ql + rng.integers(0, 90, size=n)).tolist()
    win = [int(w) if rng.random() < 0.5 else 0 for w in rng.integers(1, 60, size=n)]
    hkv = int(rng.choice([1, 2]))
    b = workloads.make_batch(ql.tolist(), kv, num_q_heads=4 * hkv, num_kv_heads=hkv,
                             head_dim=64, page_size=16, windows=win, meta_only=True)
    for part in (None, "decode", "prefill"):
        pairs, tokens, pages, nq = brute(b, part)
        c = bench.algorithmic_counts(b, part)
        assert c["pairs"] == pairs and c["kv_tokens"] == tokens
        assert c["flops"] == 4.0 * b.head_dim * b.num_q_heads * pairs
        meta = (2 * b.num_seqs + 1 + b.num_seqs) * 4
        want = tokens * hkv * b.head_dim * 2 * 2 + 2 * nq * b.num_q_heads * b.head_dim * 2 \
            + pages * 4 + meta
        assert c["bytes"] == float(want), part


def test_sliding_window_prefill_pairs():
    """8192 tokens, window 1024: key j is seen by min(1024, 8192 - j) queries."""
    b = workloads.WORKLOADS["swa_prefill"](meta_only=True)
    want = sum(min(1024, 8192 - j) for j in range(8192))
    assert want == 7864832
    c = bench.algorithmic_counts(b)
    assert c["pairs"] == want
    assert c["flops"] == 4.0 * 256 * 32 * want        # 2.577e11
