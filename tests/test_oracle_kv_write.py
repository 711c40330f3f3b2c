"""The oracle's KV-cache write ("TPU Deep Dive" slides, chapter 8, "Continuous
batching with static shapes"), pinned to something other than itself: each
sequence's cache is a dense [L, Hkv, D] array cut into pages by reshape and
placed at permuted page ids; writing the last q_len rows of the dense cache
into a pool where those slots hold zeros must rebuild the original pool
bit for bit.  Planted mistakes (off-by-one position, swapped heads, the first
instead of the last positions) each fail the pin.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle


def dense_case(seed=0, P=4, hkv=2, d=8, q_lens=(1, 3, 5, 1), kv_lens=(6, 9, 5, 13)):
    """Per-sequence dense caches, the paged pool built from them by reshape and
    a random page placement, and the new tokens' rows taken from the dense
    caches (not through the page table)."""
    rng = np.random.default_rng(seed)
    dense_k = [rng.integers(0, 1 << 16, size=(L, hkv, d), dtype=np.uint16) for L in kv_lens]
    dense_v = [rng.integers(0, 1 << 16, size=(L, hkv, d), dtype=np.uint16) for L in kv_lens]
    npages = [-(-L // P) for L in kv_lens]
    total_pages = sum(npages) + 3
    perm = rng.permutation(total_pages)
    kp = rng.integers(0, 1 << 16, size=(total_pages, P, hkv, d), dtype=np.uint16)
    vp = rng.integers(0, 1 << 16, size=(total_pages, P, hkv, d), dtype=np.uint16)
    mpps = max(npages)
    pt = np.full((len(kv_lens), mpps), -1, dtype=np.int32)
    nxt = 0
    for s, L in enumerate(kv_lens):
        padded_k = np.zeros((npages[s] * P, hkv, d), dtype=np.uint16)
        padded_v = np.zeros((npages[s] * P, hkv, d), dtype=np.uint16)
        padded_k[:L] = dense_k[s]
        padded_v[:L] = dense_v[s]
        ids = perm[nxt: nxt + npages[s]]
        nxt += npages[s]
        kp[ids] = padded_k.reshape(npages[s], P, hkv, d)
        vp[ids] = padded_v.reshape(npages[s], P, hkv, d)
        pt[s, : npages[s]] = ids
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    kl = np.asarray(kv_lens, dtype=np.int32)
    k_new = np.concatenate([dense_k[s][L - ql:] for s, (L, ql) in enumerate(zip(kv_lens, q_lens))])
    v_new = np.concatenate([dense_v[s][L - ql:] for s, (L, ql) in enumerate(zip(kv_lens, q_lens))])
    # The pool as it stood before the step: the new tokens' slots hold zeros.
    kz, vz = kp.copy(), vp.copy()
    for s, (L, ql) in enumerate(zip(kv_lens, q_lens)):
        for pos in range(L - ql, L):
            kz[pt[s, pos // P], pos % P] = 0
            vz[pt[s, pos // P], pos % P] = 0
    return dict(kp=kp, vp=vp, kz=kz, vz=vz, k_new=k_new, v_new=v_new, pt=pt, cu=cu, kl=kl)


def pin_rebuilds_pool(write):
    for seed in range(3):
        c = dense_case(seed)
        kp, vp = write(c["kz"], c["vz"], c["k_new"], c["v_new"], c["pt"], c["cu"], c["kl"])
        if not (np.array_equal(kp, c["kp"]) and np.array_equal(vp, c["vp"])):
            return False
    return True


def test_write_kv_rebuilds_the_pool():
    assert pin_rebuilds_pool(oracle.write_kv)


def test_write_kv_leaves_inputs_untouched():
    c = dense_case(7)
    kz, vz = c["kz"].copy(), c["vz"].copy()
    oracle.write_kv(c["kz"], c["vz"], c["k_new"], c["v_new"], c["pt"], c["cu"], c["kl"])
    assert np.array_equal(kz, c["kz"]) and np.array_equal(vz, c["vz"])


def _mutant(kind):
    def write(k_pages, v_pages, k_new, v_new, page_table, cu, kl):
        kp, vp = k_pages.copy(), v_pages.copy()
        P, hkv = kp.shape[1], kp.shape[2]
        for s in range(kl.shape[0]):
            ql = int(cu[s + 1] - cu[s])
            for i in range(ql):
                t = int(cu[s]) + i
                pos = int(kl[s]) - ql + i
                if kind == "off_by_one":
                    pos = int(kl[s]) - ql + i - 1 if i > 0 else pos
                if kind == "first_positions":
                    pos = i
                page = int(page_table[s, pos // P])
                for g in range(hkv):
                    gs = (hkv - 1 - g) if kind == "swap_heads" else g
                    kp[page, pos % P, gs] = k_new[t, g]
                    vp[page, pos % P, gs] = v_new[t, g]
        return kp, vp
    return write


@pytest.mark.parametrize("kind", ["off_by_one", "first_positions", "swap_heads"])
def test_pin_catches_planted_mistakes(kind):
    assert not pin_rebuilds_pool(_mutant(kind))
