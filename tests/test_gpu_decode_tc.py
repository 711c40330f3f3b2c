"""GPU parity of the tensor-core split-KV decode kernel (decode_kernel = 2)
against the CPU oracle, and against the CUDA-core decode kernel
(decode_kernel = 1), through the C ABI.

Same tolerances as test_gpu_parity.py (bf16: max 2e-2, mean 2e-3 against the
oracle in fp32 accumulation); `out` is NaN-filled before every call and the
`poisoned` cases put NaN in every pool slot no query sees.  The cases cover
what the kernel's tiling has to get right: pages of 16 to 256 tokens (boxes
of one page or less, stages spanning several pages), windows and lengths off
16-key boundaries (the V rows a box brings in past either end of the visible
keys), sequences cut across CTAs (fp32 partials and the combine), head_dim
128 and 256, G = 1 to 8 with fewer and more than 16 query heads, and a bad
page id.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ragged_paged_attention_rpa_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3
TC, MMA = 2, 1
BF16_NAN = np.uint16(0x7FC0)


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def run_gpu(b, **plan_kw):
    db = binding.Batch(b)
    plan = db.plan(**plan_kw)
    ws = binding.alloc_workspace(plan)
    db.out.fill_(float("nan"))
    out = db.forward(plan, ws)
    err = binding.rpa_get_device_error(ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().reshape(-1, b.head_dim).astype(np.float64), err, plan


def oracle_rows(b):
    return oracle.attention(b.q, b.k_pages, b.v_pages, b.page_table, b.cu_q_lens,
                            b.kv_lens, b.window, b.sm_scale, precision=32)


def assert_bf16_close(got, ref, what=""):
    e = np.abs(got - ref)
    assert np.isfinite(got).all(), what + ": non-finite output"
    assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN, \
        "%s: max %.3g mean %.3g" % (what, e.max(), e.mean())


def poisoned(b):
    """NaN in every K and V slot that no query of the batch sees."""
    seen = np.zeros((b.num_pages, b.page_size), dtype=bool)
    for s in range(b.num_seqs):
        ql = int(b.cu_q_lens[s + 1] - b.cu_q_lens[s])
        if ql == 0:
            continue
        L = int(b.kv_lens[s])
        w = 0 if b.window is None else int(b.window[s])
        lo = max(0, L - ql - w + 1) if w > 0 else 0
        j = np.arange(lo, L)
        seen[b.page_table[s, j // b.page_size], j % b.page_size] = True
    k, v = b.k_pages.copy(), b.v_pages.copy()
    k[~seen] = BF16_NAN
    v[~seen] = BF16_NAN
    return workloads.Batch(**{**b.__dict__, "k_pages": k, "v_pages": v})


# (kv_lens, Hq, Hkv, D, P, windows): decode batches (every q_len 1)
CASES = [
    ([1, 2, 15, 16, 17, 127, 128, 129, 700, 2047], 8, 1, 256, 128, None),
    ([3, 64, 65, 200, 1000, 5, 40, 333], 8, 2, 128, 32, [0, 16, 0, 100, 0, 2, 9, 77]),
    ([2000, 37, 513, 90, 1500], 2, 2, 256, 16, [1000, 0, 64, 0, 129]),
    ([129, 4097, 64, 1, 900], 16, 2, 128, 64, None),
    ([300, 1200, 4000, 77], 32, 4, 256, 256, [0, 517, 0, 33]),
    ([50, 600, 1800], 6, 2, 128, 16, [0, 31, 0]),           # G = 3
    ([999, 1001, 17, 2500], 4, 4, 256, 128, [255, 0, 0, 1000]),  # G = 1
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_decode_tc_small(case):
    kv, hq, hkv, d, p, win = CASES[case]
    b = poisoned(workloads.make_batch([1] * len(kv), kv, num_q_heads=hq, num_kv_heads=hkv,
                                      head_dim=d, page_size=p, windows=win, seed=3100 + case))
    ref = oracle_rows(b)
    got, err, plan = run_gpu(b, decode_kernel=TC)
    assert err == 0 and plan.info()["decode_kernel"] == TC
    assert_bf16_close(got, ref, "tc case %d" % case)
    mma, err, plan = run_gpu(b, decode_kernel=MMA)
    assert err == 0 and plan.info()["decode_kernel"] == MMA
    assert_bf16_close(mma, ref, "mma case %d" % case)


@pytest.mark.parametrize("split", [16, 48, 128, 448])
def test_decode_tc_split_parts(split):
    """Short CTA ranges: most sequences are cut across several CTAs, whose
    fp32 partials the combine kernel merges; ranges start and end inside
    128-key tiles."""
    kv, hq, hkv, d, p, win = CASES[2]
    b = poisoned(workloads.make_batch([1] * len(kv), kv, num_q_heads=hq, num_kv_heads=hkv,
                                      head_dim=d, page_size=p, windows=win, seed=3200))
    got, err, plan = run_gpu(b, decode_kernel=TC, kv_split=split)
    assert err == 0 and plan.info()["max_splits"] > 1
    assert_bf16_close(got, oracle_rows(b), "split %d" % split)


def test_decode_tc_workload_poisoned():
    """The full decode batch (128 sequences, D 256, G 8), NaN in every
    unseen slot, on both kernels."""
    b = poisoned(workloads.decode_batch(seed=1))
    ref = oracle_rows(b)
    for kernel in (TC, MMA):
        got, err, plan = run_gpu(b, decode_kernel=kernel)
        assert err == 0 and plan.info()["decode_kernel"] == kernel
        assert_bf16_close(got, ref, "decode kernel %d" % kernel)


def test_decode_tc_many_short_sequences():
    rng = np.random.default_rng(5)
    n = 2500
    kv = rng.integers(1, 65, size=n).tolist()
    b = workloads.make_batch([1] * n, kv, num_q_heads=8, num_kv_heads=2, head_dim=128,
                             page_size=16, windows=[0 if i % 3 else 9 for i in range(n)],
                             seed=91)
    got, err, plan = run_gpu(b, decode_kernel=TC)
    assert err == 0 and plan.info()["decode_kernel"] == TC
    assert_bf16_close(got, oracle_rows(b), "many short decode sequences")


def test_decode_tc_mixed_workload():
    """The mixed batch with its decode part on the tensor-core kernel, beside
    the prefill grid."""
    b = poisoned(workloads.mixed_batch(seed=4))
    got, err, plan = run_gpu(b, decode_kernel=TC)
    assert err == 0 and plan.info()["decode_kernel"] == TC
    assert_bf16_close(got, oracle_rows(b), "mixed")


def test_decode_tc_bad_page_id_sets_the_error_word():
    b = workloads.decode_batch(seed=6, num_seqs=8, pool_pages=160)
    db = binding.Batch(b)
    plan = db.plan(decode_kernel=TC)
    ws = binding.alloc_workspace(plan)
    pt = db.page_table.clone()
    pt[3, 0] = b.num_pages + 7          # outside the pool: the kernel must skip it
    binding.rpa_forward(db.q, db.k_pages, db.v_pages, pt, db.cu_q_lens, db.kv_lens,
                        db.window, b.sm_scale, db.out, plan, ws)
    assert binding.rpa_get_device_error(ws) == binding.RPA_DEVERR_PAGE_ID
    db.forward(plan, ws)
    assert binding.rpa_get_device_error(ws) == 0
    got = db.out.float().cpu().numpy().reshape(-1, b.head_dim).astype(np.float64)
    assert_bf16_close(got, oracle_rows(b))


def test_decode_tc_page_permutation_is_bitwise_invisible():
    b = workloads.decode_batch(seed=5, num_seqs=32, pool_pages=600)
    got, _, _ = run_gpu(b, decode_kernel=TC)
    perm = np.random.default_rng(9).permutation(b.num_pages)
    k2 = np.empty_like(b.k_pages)
    v2 = np.empty_like(b.v_pages)
    k2[perm] = b.k_pages
    v2[perm] = b.v_pages
    pt2 = np.where(b.page_table >= 0, perm[np.maximum(b.page_table, 0)], -1).astype(np.int32)
    b2 = workloads.Batch(**{**b.__dict__, "k_pages": k2, "v_pages": v2, "page_table": pt2})
    got2, _, _ = run_gpu(b2, decode_kernel=TC)
    assert np.array_equal(got, got2)
