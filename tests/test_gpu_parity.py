"""GPU parity: librpa (through its C ABI) against the CPU oracle.

Tolerances:
  * bf16 in/out: max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3 over
    the compared outputs, the oracle in fp32 accumulation, unrounded;
  * fp32 debug build: max |gpu - oracle| / max |oracle| <= 1e-5 (normwise; an
    elementwise relative bound is meaningless near zero outputs).
Every test compares every output row, the five full-size workloads included;
`out` is filled with NaN before each call, so a row the kernels never write
fails.  Pool slots that no query of the batch sees (free slots past a
sequence's last key, keys before every query's window, pages no sequence owns)
are set to NaN in the `poisoned` tests: the definition never reads them, so
neither may the result depend on them.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ragged_paged_attention_rpa_gb300 import binding, build, workloads
from ragged_paged_attention_rpa_gb300.binding import RPA_PATH_SIMT, RPA_PATH_TC

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, F32_NORMWISE = 2e-2, 2e-3, 1e-5


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


def oracle_rows(b, rows=None):
    return oracle.attention(b.q, b.k_pages, b.v_pages, b.page_table, b.cu_q_lens,
                            b.kv_lens, b.window, b.sm_scale, rows=rows, precision=32)


def assert_bf16_close(got, ref, what=""):
    e = np.abs(got - ref)
    assert np.isfinite(got).all(), what + ": non-finite output"
    assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN, \
        "%s: max %.3g mean %.3g" % (what, e.max(), e.mean())


BF16_NAN = np.uint16(0x7FC0)


def unseen_slots(b):
    """[num_pages, page_size] mask of the pool slots no query of the batch
    sees: for sequence s the visible keys of its queries together are
    max(0, L - q_len - W + 1) .. L - 1 (W <= 0: from 0)."""
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
    return ~seen


def poisoned(b):
    """The batch with NaN in every K and V slot no query sees."""
    mask = unseen_slots(b)
    k, v = b.k_pages.copy(), b.v_pages.copy()
    nan = BF16_NAN if k.dtype == np.uint16 else np.float32("nan")
    k[mask] = nan
    v[mask] = nan
    return workloads.Batch(**{**b.__dict__, "k_pages": k, "v_pages": v})


# ---------------------------------------------------------------- small cases

SMALL = [
    # (q_lens, kv_lens, Hq, Hkv, D, P, windows)
    ([5, 1, 0, 17, 1, 33], [9, 33, 4, 40, 1, 300], 4, 2, 64, 16, [0, 5, 0, 7, 1, 64]),
    ([1] * 9, [1, 2, 15, 16, 17, 127, 128, 129, 700], 8, 1, 256, 128, None),
    ([1] * 6 + [20], [3, 64, 65, 200, 1000, 5, 40], 8, 2, 128, 32, [0, 16, 0, 100, 0, 2, 9]),
    ([1, 1, 1, 70], [2000, 37, 513, 90], 2, 2, 256, 16, [1000, 0, 64, 0]),
    ([1, 1, 64, 1], [129, 4097, 64, 1], 16, 2, 64, 64, None),
    ([1, 3, 1], [40, 20, 7], 4, 1, 64, 8, [0, 0, 3]),          # 8-token pages: CUDA-core path
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_ragged_bf16(case):
    ql, kv, hq, hkv, d, p, win = SMALL[case]
    b = workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=p, windows=win, pool_pages=None, seed=100 + case)
    got, err, plan = run_gpu(b)
    assert err == 0
    assert_bf16_close(got, oracle_rows(b), "case %d" % case)


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_ragged_f32_debug(case):
    ql, kv, hq, hkv, d, p, win = SMALL[case]
    b = workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=p, windows=win, seed=200 + case, dtype="f32")
    got, err, plan = run_gpu(b)
    assert err == 0 and plan.info()["path"] == RPA_PATH_SIMT
    ref = oracle_rows(b)
    nw = np.abs(got - ref).max() / np.abs(ref).max()
    assert nw <= F32_NORMWISE, nw


def test_simt_path_bf16_matches_oracle():
    ql, kv, hq, hkv, d, p, win = SMALL[2]
    b = workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=p, windows=win, seed=300)
    got, err, plan = run_gpu(b, path=RPA_PATH_SIMT)
    assert err == 0 and plan.info()["path"] == RPA_PATH_SIMT
    assert_bf16_close(got, oracle_rows(b))


def test_tiny_prefill_workload():
    b = workloads.tiny_prefill(seed=0)
    got, err, _ = run_gpu(b)
    assert err == 0
    assert_bf16_close(got, oracle_rows(b), "tiny prefill")


def test_empty_batch_is_a_no_op():
    b = workloads.make_batch([0, 0], [5, 0], num_q_heads=8, num_kv_heads=1, head_dim=256,
                             page_size=128, seed=1)
    db = binding.Batch(b)
    plan = db.plan()
    ws = binding.alloc_workspace(plan)
    db.forward(plan, ws)
    assert binding.rpa_get_device_error(ws) == 0


# ---------------------------------------------------------------- prefill (tensor cores)

PREFILL = [
    # (q_lens, kv_lens, Hq, Hkv, D, P, windows)
    ([200, 129, 64], [300, 129, 1000], 4, 4, 128, 128, [100, 0, 0]),      # G = 1
    ([1000], [1000], 4, 2, 256, 128, [0]),                                 # G = 2 causal
    ([1000], [1000], 4, 2, 256, 128, [256]),                               # G = 2 window
    ([100, 1, 37], [400, 50, 37], 8, 1, 256, 128, [64, 0, 1024]),          # G = 8, chunked
    ([70, 33, 2], [70, 90, 2], 8, 2, 64, 16, [0, 20, 0]),                  # G = 4, P = 16
    ([45, 80], [45, 300], 6, 2, 128, 64, [0, 33]),                         # G = 3
    ([40, 17], [100, 17], 16, 1, 64, 32, [0, 5]),                          # G = 16
    ([130, 65], [130, 2000], 2, 2, 256, 16, [0, 0]),                       # G = 1, P = 16
    ([300, 150], [600, 150], 8, 2, 64, 128, [100, 70]),                    # D = 64, P = 128, windows
]


@pytest.mark.parametrize("case", range(len(PREFILL)))
def test_prefill_tc_small(case):
    ql, kv, hq, hkv, d, p, win = PREFILL[case]
    b = workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=p, windows=win, seed=400 + case)
    got, err, plan = run_gpu(b)
    info = plan.info()
    assert err == 0 and info["path"] == RPA_PATH_TC and info["num_prefill_items"] > 0
    assert_bf16_close(got, oracle_rows(b), "prefill case %d" % case)


def test_decode_many_short_sequences():
    """Thousands of short decode sequences: several launches, many sequences
    per CTA range, cut sequences merged by the combine kernel."""
    rng = np.random.default_rng(5)
    n = 2500
    kv = rng.integers(1, 65, size=n).tolist()
    b = workloads.make_batch([1] * n, kv, num_q_heads=8, num_kv_heads=2, head_dim=128,
                             page_size=16, windows=[0 if i % 3 else 9 for i in range(n)],
                             seed=91)
    got, err, plan = run_gpu(b)
    assert err == 0 and plan.info()["path"] == RPA_PATH_TC
    assert plan.info()["num_decode_seqs"] == n
    assert_bf16_close(got, oracle_rows(b), "many short decode sequences")


@pytest.mark.parametrize("case", [0, 2, 3, 5, 7])
def test_prefill_sm_pairs(case):
    """The SM-pair prefill kernel (one M = 256 MMA over two query blocks)."""
    ql, kv, hq, hkv, d, p, win = PREFILL[case]
    b = workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=p, windows=win, seed=600 + case)
    got, err, plan = run_gpu(b, prefill_pairs=2)
    info = plan.info()
    assert err == 0 and info["prefill_pairs"] == 1
    assert info["prefill_ctas"] % 2 == 0
    assert_bf16_close(got, oracle_rows(b), "pair prefill case %d" % case)


@pytest.mark.parametrize("q_block", [64, 32, 16, 8])
def test_prefill_q_block_invariance(q_block):
    """The query block changes scheduling, not the result."""
    b = workloads.make_batch([700, 300], [700, 900], num_q_heads=4, num_kv_heads=2,
                             head_dim=256, page_size=128, windows=[0, 128], seed=77)
    got, err, plan = run_gpu(b, q_block=q_block)
    assert err == 0 and plan.info()["q_block"] == q_block
    assert_bf16_close(got, oracle_rows(b), "q_block %d" % q_block)


def test_prefill_tc_and_simt_agree():
    b = workloads.make_batch([300], [500], num_q_heads=8, num_kv_heads=2, head_dim=128,
                             page_size=64, windows=[200], seed=78)
    tc, err1, _ = run_gpu(b, path=RPA_PATH_TC)
    simt, err2, _ = run_gpu(b, path=RPA_PATH_SIMT)
    assert err1 == 0 and err2 == 0
    assert np.abs(tc - simt).max() <= 2 * BF16_MAX


# ---------------------------------------------------------------- decode


@pytest.fixture(scope="module")
def decode_case():
    b = workloads.decode_batch(seed=1)
    return b, oracle_rows(b)


def test_decode_workload_full(decode_case):
    b, ref = decode_case
    got, err, plan = run_gpu(b)
    assert err == 0 and plan.info()["path"] == RPA_PATH_TC
    assert_bf16_close(got, ref, "decode")


@pytest.mark.parametrize("split", [64, 128, 448, 2048])
def test_decode_split_invariance(decode_case, split):
    """The split length changes scheduling, not the result."""
    b, ref = decode_case
    got, err, plan = run_gpu(b, kv_split=split)
    assert err == 0 and plan.info()["kv_split"] == split
    assert_bf16_close(got, ref, "split %d" % split)


def test_decode_simt_and_tc_agree(decode_case):
    b, ref = decode_case
    simt, err, _ = run_gpu(b, path=RPA_PATH_SIMT)
    assert err == 0
    assert_bf16_close(simt, ref, "simt decode")


def test_page_permutation_is_bitwise_invisible():
    b = workloads.decode_batch(seed=5, num_seqs=32, pool_pages=600)
    got, _, _ = run_gpu(b)
    perm = np.random.default_rng(9).permutation(b.num_pages)
    k2 = np.empty_like(b.k_pages)
    v2 = np.empty_like(b.v_pages)
    k2[perm] = b.k_pages
    v2[perm] = b.v_pages
    pt2 = np.where(b.page_table >= 0, perm[np.maximum(b.page_table, 0)], -1).astype(np.int32)
    b2 = workloads.Batch(**{**b.__dict__, "k_pages": k2, "v_pages": v2, "page_table": pt2})
    got2, _, _ = run_gpu(b2)
    assert np.array_equal(got, got2)


def test_bad_page_id_sets_the_error_word_without_faulting():
    b = workloads.decode_batch(seed=6, num_seqs=8, pool_pages=160)
    db = binding.Batch(b)
    plan = db.plan()
    ws = binding.alloc_workspace(plan)
    pt = db.page_table.clone()
    pt[3, 0] = b.num_pages + 7          # outside the pool: the kernel must skip it
    binding.rpa_forward(db.q, db.k_pages, db.v_pages, pt, db.cu_q_lens, db.kv_lens,
                        db.window, b.sm_scale, db.out, plan, ws)
    assert binding.rpa_get_device_error(ws) == binding.RPA_DEVERR_PAGE_ID
    # The error word was cleared by the read, and a good call still works.
    db.forward(plan, ws)
    assert binding.rpa_get_device_error(ws) == 0
    got = db.out.float().cpu().numpy().reshape(-1, b.head_dim).astype(np.float64)
    assert_bf16_close(got, oracle_rows(b))


# ---------------------------------------------------------------- the full-size workloads


@pytest.mark.parametrize("name", ["swa_prefill", "causal_prefill"])
def test_prefill_workloads_full(name):
    """The 8192-token prefills (32 q / 16 kv heads, D 256), every output row."""
    b = workloads.WORKLOADS[name]()
    got, err, _ = run_gpu(b)
    assert err == 0
    assert_bf16_close(got, oracle_rows(b), name)


def test_prefill_l2_groups_change_order_not_bits():
    """The causal 8k prefill's dynamic list in four L2-sized groups of KV
    heads (the default) and longest first over all heads (prefill_grouping =
    -1) give the same bits: the grouping only reorders whole items."""
    b = workloads.WORKLOADS["causal_prefill"]()
    grouped, err, plan = run_gpu(b)
    assert err == 0 and plan.info()["prefill_groups"] == 4
    flat, err, fplan = run_gpu(b, prefill_grouping=-1)
    assert err == 0 and fplan.info()["prefill_groups"] == 1
    assert np.array_equal(grouped, flat)


@pytest.fixture(scope="module")
def mixed_case():
    b = poisoned(workloads.mixed_batch(seed=4))
    return b, oracle_rows(b)


def test_mixed_workload_full(mixed_case):
    """512 decode sequences and 4 chunked prefills of 2048 tokens, half of
    them windowed, every output row, with NaN in every slot no query sees."""
    b, ref = mixed_case
    got, err, plan = run_gpu(b)
    assert err == 0
    info = plan.info()
    assert info["num_decode_seqs"] == 512 and info["num_prefill_seqs"] == 4
    assert_bf16_close(got, ref, "mixed")


# ---------------------------------------------------------------- multi-token decode

SPEC = [
    # (spec tokens, Hq, Hkv, D, P): spec x G query rows per KV head
    (8, 8, 1, 256, 128),     # 64 rows, the decode batch's heads
    (4, 16, 2, 128, 64),     # 32 rows
    (2, 8, 1, 64, 16),       # 16 rows
    (16, 8, 1, 256, 128),    # 128 rows: one full tile
]


@pytest.mark.parametrize("case", range(len(SPEC)))
def test_multi_token_decode(case):
    """Speculative decode: every sequence verifies `spec` drafted tokens in one
    step (causal among themselves, after the cached prefix); the tensor-core
    kernel packs spec x G rows of one KV head into its M dimension."""
    spec, hq, hkv, d, p = SPEC[case]
    rng = np.random.default_rng(800 + case)
    n = 24
    kv = rng.integers(spec, 1500, size=n).tolist()
    win = [0 if i % 3 else 300 for i in range(n)]
    b = workloads.make_batch([spec] * n, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=p, windows=win, seed=810 + case)
    got, err, plan = run_gpu(b)
    info = plan.info()
    assert err == 0 and info["path"] == RPA_PATH_TC and info["num_prefill_seqs"] == n
    assert_bf16_close(got, oracle_rows(b), "multi-token decode case %d" % case)


def test_spec_decode_workload_full():
    b = workloads.WORKLOADS["spec_decode"]()
    got, err, _ = run_gpu(b)
    assert err == 0
    assert_bf16_close(got, oracle_rows(b), "spec_decode")


@pytest.mark.parametrize("case,tiles", [(0, 2), (1, 2), (2, 1), (3, 1), (5, 1), (7, 2), (8, 1)])
def test_prefill_split_parts(case, tiles):
    """Prefill items cut into parts of one or two key tiles (forced), each
    part's fp32 partial merged by the combine kernel, against the oracle."""
    ql, kv, hq, hkv, d, p, win = PREFILL[case]
    b = workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=p, windows=win, seed=1000 + case)
    got, err, plan = run_gpu(b, prefill_split=tiles)
    info = plan.info()
    assert err == 0 and info["prefill_split_items"] > 0
    assert_bf16_close(got, oracle_rows(b), "split prefill case %d" % case)


# ---------------------------------------------------------------- unseen slots hold NaN


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_ragged_poisoned(case):
    ql, kv, hq, hkv, d, p, win = SMALL[case]
    b = poisoned(workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                      page_size=p, windows=win, pool_pages=None,
                                      seed=1300 + case))
    got, err, plan = run_gpu(b)
    assert err == 0
    assert_bf16_close(got, oracle_rows(b), "poisoned case %d" % case)


@pytest.mark.parametrize("case", range(len(PREFILL)))
def test_prefill_tc_poisoned(case):
    ql, kv, hq, hkv, d, p, win = PREFILL[case]
    b = poisoned(workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                      page_size=p, windows=win, seed=1400 + case))
    assert unseen_slots(b).any()
    got, err, plan = run_gpu(b)
    assert err == 0 and plan.info()["path"] == RPA_PATH_TC
    assert_bf16_close(got, oracle_rows(b), "poisoned prefill case %d" % case)


@pytest.mark.parametrize("case", [0, 2, 3, 5, 7])
def test_prefill_sm_pairs_poisoned(case):
    ql, kv, hq, hkv, d, p, win = PREFILL[case]
    b = poisoned(workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                      page_size=p, windows=win, seed=1500 + case))
    got, err, plan = run_gpu(b, prefill_pairs=2)
    assert err == 0 and plan.info()["prefill_pairs"] == 1
    assert_bf16_close(got, oracle_rows(b), "poisoned pair prefill case %d" % case)


@pytest.mark.parametrize("case,tiles", [(2, 1), (3, 1), (7, 2), (8, 1)])
def test_prefill_split_parts_poisoned(case, tiles):
    ql, kv, hq, hkv, d, p, win = PREFILL[case]
    b = poisoned(workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                      page_size=p, windows=win, seed=1600 + case))
    got, err, plan = run_gpu(b, prefill_split=tiles)
    assert err == 0 and plan.info()["prefill_split_items"] > 0
    assert_bf16_close(got, oracle_rows(b), "poisoned split prefill case %d" % case)


def test_decode_workload_poisoned():
    """The decode batch with NaN in the free slots of every last page, before
    every window and in the 2900-odd pool pages no sequence owns."""
    b = poisoned(workloads.decode_batch(seed=1))
    got, err, plan = run_gpu(b)
    assert err == 0
    assert_bf16_close(got, oracle_rows(b), "poisoned decode")
    windowed = poisoned(workloads.make_batch([1] * 40, list(range(100, 4100, 100)),
                                             num_q_heads=8, num_kv_heads=1, head_dim=256,
                                             page_size=128, windows=[300 + 7 * i for i in range(40)],
                                             seed=17))
    got, err, _ = run_gpu(windowed)
    assert err == 0
    assert_bf16_close(got, oracle_rows(windowed), "poisoned windowed decode")


# ---------------------------------------------------------------- query blocks of two tiles


@pytest.mark.parametrize("q_block", [128, 64])
def test_prefill_q_block_on_sm_pairs(q_block):
    """A 128-token query block at G = 2 (two 128-row tiles) runs on SM pairs;
    same result as any other block size."""
    b = workloads.make_batch([700, 300], [700, 900], num_q_heads=4, num_kv_heads=2,
                             head_dim=256, page_size=128, windows=[0, 128], seed=77)
    got, err, plan = run_gpu(b, q_block=q_block, prefill_pairs=2)
    info = plan.info()
    assert err == 0 and info["q_block"] == q_block and info["prefill_pairs"] == 1
    assert_bf16_close(got, oracle_rows(b), "q_block %d on pairs" % q_block)


# ---------------------------------------------------------------- dynamic item order


@pytest.mark.parametrize("case", [0, 2, 5, 7])
def test_prefill_dynamic_items_match_fixed_lists_bitwise(case):
    """Items taken dynamically (work counter in the workspace header) give
    the same bits as the planner's fixed per-CTA lists: each item's
    arithmetic does not depend on which CTA runs it.  Two calls in a row on
    one workspace check that the counter is left at zero."""
    ql, kv, hq, hkv, d, p, win = PREFILL[case]
    b = poisoned(workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                      page_size=p, windows=win, seed=1700 + case))
    db = binding.Batch(b)
    plan = db.plan()
    assert plan.info()["prefill_dynamic"] == 1
    ws = binding.alloc_workspace(plan)
    outs = []
    for _ in range(2):
        db.out.fill_(float("nan"))
        outs.append(db.forward(plan, ws).clone())
    assert binding.rpa_get_device_error(ws) == 0
    counters = ws[64:72].view(torch.int32).cpu().tolist()
    assert counters == [0, 0]
    fixed, err, fplan = run_gpu(b, prefill_dynamic=-1)
    assert err == 0 and fplan.info()["prefill_dynamic"] == 0
    got = outs[0].float().cpu().numpy().reshape(-1, b.head_dim).astype(np.float64)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert np.array_equal(got, fixed)
    assert_bf16_close(got, oracle_rows(b), "dynamic prefill case %d" % case)
