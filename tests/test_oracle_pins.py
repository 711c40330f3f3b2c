"""Pins for the CPU oracle: it is checked against things other than itself.

Each pin is a function returning (ok, detail) so that ``test_oracle_mutants``
can run the same pins against copies of the oracle with a planted mistake and
show that every plausible mistake fails at least one of them.

Pins (none of them re-calls the oracle's own formula):
  * hand-derived closed forms stored under tests/golden/ (cited there);
  * a dense brute force in numpy float64 over contiguous (un-paged) K/V with an
    explicit mask matrix, on tiny ragged batches;
  * invariants: permuting physical pages, window >= L, GQA = MHA with
    replicated KV heads, a single visible key, rows summing to 1, sm_scale = 0
    giving the mean of the visible values;
  * the window semantics of "Chasing speed of light on TPU v6e", section
    "Attention": in an 8192-token sequence with a 1024 window every key is seen
    by the 1024 queries that follow it (fewer at the end), 7,864,832 pairs.
"""

from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import oracle
from ragged_paged_attention_rpa_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def bits_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bits(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def run(b, lib=None, precision=32, window="batch", **kw):
    win = b.window if isinstance(window, str) else window
    return oracle.attention(b.q, b.k_pages, b.v_pages, b.page_table, b.cu_q_lens,
                            b.kv_lens, win, b.sm_scale, precision=precision,
                            lib_path=lib, **kw)


def dense_reference(b, window="batch"):
    """Float64 brute force: gather each sequence's pages into contiguous K/V,
    build an explicit [q_len, L] visibility matrix, softmax(Q K^T s + mask) V."""
    win = b.window if isinstance(window, str) else window
    to64 = (lambda a: bits_to_f32(a).astype(np.float64)) if b.dtype == "bf16" else \
        (lambda a: a.astype(np.float64))
    q, k, v = to64(b.q), to64(b.k_pages), to64(b.v_pages)
    hq, hkv, d, p = b.num_q_heads, b.num_kv_heads, b.head_dim, b.page_size
    out = np.zeros((b.total_q, hq, d))
    for s in range(b.num_seqs):
        L = int(b.kv_lens[s])
        t0, t1 = int(b.cu_q_lens[s]), int(b.cu_q_lens[s + 1])
        ql = t1 - t0
        if ql == 0:
            continue
        n_pages = -(-L // p)
        kc = k[b.page_table[s, :n_pages]].reshape(n_pages * p, hkv, d)[:L]
        vc = v[b.page_table[s, :n_pages]].reshape(n_pages * p, hkv, d)[:L]
        pos = np.arange(L - ql, L)[:, None]
        j = np.arange(L)[None, :]
        w = 0 if win is None else int(win[s])
        mask = (j <= pos) & ((w <= 0) | (pos - j < w))
        for h in range(hq):
            g = h // (hq // hkv)
            sc = (q[t0:t1, h, :] @ kc[:, g, :].T) * b.sm_scale
            sc = np.where(mask, sc, -np.inf)
            e = np.exp(sc - sc.max(axis=1, keepdims=True))
            out[t0:t1, h, :] = (e / e.sum(axis=1, keepdims=True)) @ vc[:, g, :]
    return out.reshape(-1, d)


def normwise(a, ref):
    return float(np.abs(a - ref).max() / max(np.abs(ref).max(), 1e-300))


def tiny_batches():
    """Small ragged batches covering decode, prefill, chunked prefill, windows,
    GQA, empty sequences and page sizes 4 and 16."""
    yield workloads.make_batch([5, 1, 0, 17, 1], [9, 33, 4, 40, 1], num_q_heads=4,
                               num_kv_heads=2, head_dim=16, page_size=4,
                               windows=[0, 5, 0, 7, 1], pool_pages=40, seed=11,
                               name="ragged_p4")
    yield workloads.make_batch([64, 3], [64, 50], num_q_heads=8, num_kv_heads=1,
                               head_dim=32, page_size=16, windows=[16, 0],
                               pool_pages=12, seed=12, name="mqa_p16")
    yield workloads.make_batch([1, 1, 1, 1], [1, 16, 17, 64], num_q_heads=2,
                               num_kv_heads=2, head_dim=8, page_size=16,
                               pool_pages=9, seed=13, name="decode_mha_p16")


# ---------------------------------------------------------------- pins


def pin_golden(lib=None):
    cases = json.load(open(GOLDEN))["cases"]
    worst = 0.0
    for c in cases:
        q = np.array(c["q"], dtype=np.float32)
        k = np.array(c["k_pages"], dtype=np.float32)
        v = np.array(c["v_pages"], dtype=np.float32)
        win = None if c["window"] is None else np.array(c["window"], dtype=np.int32)
        exp = np.array(c["expected"], dtype=np.float64).reshape(-1, c["head_dim"])
        for ins in ((q, k, v), (f32_to_bits(q), f32_to_bits(k), f32_to_bits(v))):
            for prec, tol in ((32, 1e-6), (64, 1e-14)):
                got = oracle.attention(*ins, c["page_table"], c["cu_q_lens"],
                                       c["kv_lens"], win, c["sm_scale"],
                                       precision=prec, lib_path=lib)
                err = float(np.abs(got - exp).max())
                worst = max(worst, err)
                if err > tol:
                    return False, "%s prec %d: err %.3g" % (c["name"], prec, err)
    return True, "worst %.3g" % worst


def pin_brute_force(lib=None):
    for b in list(tiny_batches()) + [workloads.tiny_prefill(seed=0)]:
        ref = dense_reference(b)
        e32 = normwise(run(b, lib, 32), ref)
        e64 = normwise(run(b, lib, 64), ref)
        if not (e32 <= 1e-6 and e64 <= 1e-12):
            return False, "%s: fp32 %.3g fp64 %.3g" % (b.name, e32, e64)
    return True, "ok"


def pin_page_permutation(lib=None):
    for b in tiny_batches():
        base = run(b, lib)
        rng = np.random.default_rng(5)
        perm = rng.permutation(b.num_pages)          # old page p -> new page perm[p]
        k2 = np.empty_like(b.k_pages)
        v2 = np.empty_like(b.v_pages)
        k2[perm] = b.k_pages
        v2[perm] = b.v_pages
        pt2 = np.where(b.page_table >= 0, perm[np.maximum(b.page_table, 0)], -1)
        got = oracle.attention(b.q, k2, v2, pt2.astype(np.int32), b.cu_q_lens,
                               b.kv_lens, b.window, b.sm_scale, lib_path=lib)
        if not np.array_equal(got, base):
            return False, b.name
    return True, "ok"


def pin_window_ge_len(lib=None):
    for b in tiny_batches():
        full = run(b, lib, window=None)
        big = run(b, lib, window=np.maximum(b.kv_lens, 1).astype(np.int32))
        bigger = run(b, lib, window=(b.kv_lens + 1000).astype(np.int32))
        if not (np.array_equal(full, big) and np.array_equal(full, bigger)):
            return False, b.name
    return True, "ok"


def pin_single_key(lib=None):
    # Window 1: each query sees only its own key, so out = v at its position.
    b = next(iter(tiny_batches()))
    got = run(b, lib, window=np.ones(b.num_seqs, dtype=np.int32)).reshape(
        b.total_q, b.num_q_heads, b.head_dim)
    vf = bits_to_f32(b.v_pages)
    G = b.num_q_heads // b.num_kv_heads
    for s in range(b.num_seqs):
        ql = int(b.cu_q_lens[s + 1] - b.cu_q_lens[s])
        for i in range(ql):
            pos = int(b.kv_lens[s]) - ql + i
            page = b.page_table[s, pos // b.page_size]
            for h in range(b.num_q_heads):
                want = vf[page, pos % b.page_size, h // G]
                if not np.array_equal(got[b.cu_q_lens[s] + i, h], want.astype(np.float64)):
                    return False, "seq %d query %d head %d" % (s, i, h)
    # Position 0 of a prefill sees exactly one key even without a window.
    t = workloads.tiny_prefill(seed=3)
    got0 = run(t, lib, rows=np.arange(t.num_q_heads))
    want0 = bits_to_f32(t.v_pages)[t.page_table[0, 0], 0, 0].astype(np.float64)
    if not all(np.array_equal(got0[h], want0) for h in range(t.num_q_heads)):
        return False, "position 0"
    return True, "ok"


def pin_rows_sum_to_one(lib=None):
    for b in tiny_batches():
        for r in range(0, b.total_q * b.num_q_heads, 3):
            p, lo, hi = oracle.softmax_row(b.q, b.k_pages, b.v_pages, b.page_table,
                                           b.cu_q_lens, b.kv_lens, b.window,
                                           b.sm_scale, r, lib_path=lib)
            if abs(p.sum() - 1.0) > 1e-6 or np.any(p < 0):
                return False, "%s row %d sum %.9f" % (b.name, r, p.sum())
    return True, "ok"


def pin_zero_scale_mean(lib=None):
    for b in tiny_batches():
        b0 = workloads.Batch(**{**b.__dict__, "sm_scale": 0.0})
        got = run(b0, lib)
        # Closed form: uniform weights, so out = mean of the visible values.
        vf = bits_to_f32(b.v_pages).astype(np.float64)
        G = b.num_q_heads // b.num_kv_heads
        want = np.zeros((b.total_q, b.num_q_heads, b.head_dim))
        for s in range(b.num_seqs):
            ql = int(b.cu_q_lens[s + 1] - b.cu_q_lens[s])
            L = int(b.kv_lens[s])
            w = 0 if b.window is None else int(b.window[s])
            for i in range(ql):
                pos = L - ql + i
                lo = max(0, pos - w + 1) if w > 0 else 0
                js = np.arange(lo, pos + 1)
                pages = b.page_table[s, js // b.page_size]
                for h in range(b.num_q_heads):
                    want[b.cu_q_lens[s] + i, h] = vf[pages, js % b.page_size, h // G].mean(0)
        if normwise(got, want.reshape(-1, b.head_dim)) > 1e-6:
            return False, b.name
    return True, "ok"


def pin_gqa_equals_replicated_mha(lib=None):
    b = workloads.make_batch([7, 1, 12], [20, 9, 12], num_q_heads=6, num_kv_heads=2,
                             head_dim=8, page_size=4, windows=[3, 0, 0], pool_pages=14,
                             seed=21)
    G = 3
    k_rep = np.repeat(b.k_pages, G, axis=2)   # kv head g -> heads g*G .. g*G+G-1
    v_rep = np.repeat(b.v_pages, G, axis=2)
    gqa = run(b, lib)
    mha = oracle.attention(b.q, k_rep, v_rep, b.page_table, b.cu_q_lens, b.kv_lens,
                           b.window, b.sm_scale, lib_path=lib)
    return bool(np.array_equal(gqa, mha)), "ok"


def pin_window_pair_count(lib=None):
    """8192 tokens, window 1024: key j is seen by min(1024, 8192 - j) queries."""
    L, W = 8192, 1024
    b = workloads.make_batch([L], [L], num_q_heads=1, num_kv_heads=1, head_dim=2,
                             page_size=128, windows=[W], seed=7)
    seen = np.zeros(L, dtype=np.int64)
    for r in range(L):
        p, lo, hi = oracle.softmax_row(b.q, b.k_pages, b.v_pages, b.page_table,
                                       b.cu_q_lens, b.kv_lens, b.window, b.sm_scale,
                                       r, lib_path=lib)
        if hi != r or len(p) != hi - lo + 1:
            return False, "row %d spans %d..%d" % (r, lo, hi)
        seen[lo:hi + 1] += 1
    want = np.minimum(W, L - np.arange(L))
    if not np.array_equal(seen, want):
        return False, "coverage differs"
    if int(seen.sum()) != 7_864_832:
        return False, "pairs %d" % int(seen.sum())
    return True, "ok"


def pin_fp32_inputs_match_bf16(lib=None):
    b = next(iter(tiny_batches()))
    a = run(b, lib)
    c = oracle.attention(bits_to_f32(b.q), bits_to_f32(b.k_pages), bits_to_f32(b.v_pages),
                         b.page_table, b.cu_q_lens, b.kv_lens, b.window, b.sm_scale,
                         lib_path=lib)
    return bool(np.array_equal(a, c)), "ok"


PINS = [pin_golden, pin_brute_force, pin_page_permutation, pin_window_ge_len,
        pin_single_key, pin_rows_sum_to_one, pin_zero_scale_mean,
        pin_gqa_equals_replicated_mha, pin_window_pair_count, pin_fp32_inputs_match_bf16]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    ok, detail = pin()
    assert ok, detail


def test_rows_subset_matches_full():
    b = next(iter(tiny_batches()))
    full = run(b)
    rows = np.array([0, 5, 17, b.total_q * b.num_q_heads - 1], dtype=np.int64)
    sub = run(b, rows=rows)
    assert np.array_equal(sub, full[rows])


def test_thread_count_does_not_change_result():
    b = workloads.tiny_prefill(seed=1)
    assert np.array_equal(run(b, threads=1), run(b, threads=4))


def test_bf16_rounding_of_output():
    b = workloads.tiny_prefill(seed=2)
    out, out16 = run(b, with_bf16=True)
    ref16 = f32_to_bits(out.astype(np.float32))
    assert np.array_equal(out16, ref16)
    assert np.array_equal(oracle.round_bf16(out.astype(np.float32)), ref16)


def test_rejects_bad_metadata():
    b = next(iter(tiny_batches()))
    bad_pt = b.page_table.copy()
    bad_pt[0, 0] = b.num_pages          # page id out of range
    with pytest.raises(ValueError):
        oracle.attention(b.q, b.k_pages, b.v_pages, bad_pt, b.cu_q_lens, b.kv_lens,
                         b.window, b.sm_scale)
    bad_kv = b.kv_lens.copy()
    bad_kv[0] = 0                        # kv_len < q_len
    with pytest.raises(ValueError):
        oracle.attention(b.q, b.k_pages, b.v_pages, b.page_table, b.cu_q_lens, bad_kv,
                         b.window, b.sm_scale)
