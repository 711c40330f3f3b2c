"""rpa_forward_decode_noalloc: decode for callers that cannot allocate device
memory at call time -- code running inside a framework whose device memory is
all owned by another allocator, real-time serving loops that must not call
cudaMalloc (it may synchronise the device), plug-ins handed only the tensors
they work on.  It runs the same split-KV decode kernels as rpa_forward but
keeps their scratch in a fixed array inside librpa.

Checked through the C ABI against the CPU oracle, on two calls in a row (the
second must not depend on what the first left in the shared scratch), and
against rpa_forward with a caller workspace.  A bad page id under this entry
point sets the scratch's error word, which rpa_get_device_error(NULL) reads.
This file sorts last so that a failure here stops a -x run only after every
other test has run; it also passes alone in a fresh process.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from ragged_paged_attention_rpa_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def close(got, ref, what):
    e = np.abs(got - ref)
    assert np.isfinite(got).all(), "%s: outputs left unwritten" % what
    assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN, (what, e.max(), e.mean())


def noalloc(db, b, plan, out, page_table=None):
    binding.rpa_forward_decode_noalloc(db.q, db.k_pages, db.v_pages,
                                       db.page_table if page_table is None else page_table,
                                       db.cu_q_lens, db.kv_lens, db.window, b.sm_scale, out,
                                       plan)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().reshape(-1, b.head_dim).astype(np.float64)


def test_noalloc_decode_matches_oracle_twice():
    b = workloads.decode_batch(seed=11, num_seqs=96, pool_pages=1600)
    db = binding.Batch(b)
    plan = db.plan(kv_split=256)          # several splits per sequence: uses the scratch
    info = plan.info()
    assert info["max_splits"] > 1 and plan.workspace_bytes <= (32 << 20)
    ref = oracle.attention(b.q, b.k_pages, b.v_pages, b.page_table, b.cu_q_lens, b.kv_lens,
                           b.window, b.sm_scale, precision=32)
    ws = binding.alloc_workspace(plan)
    with_ws = db.forward(plan, ws).float().cpu().numpy().reshape(-1, b.head_dim)
    assert binding.rpa_get_device_error(ws) == 0
    assert binding.rpa_get_device_error(None) == 0
    for call in range(2):
        got = noalloc(db, b, plan, torch.full_like(db.out, float("nan")))
        close(got, ref, "call %d" % call)
        close(got, with_ws, "call %d against rpa_forward" % call)
    assert binding.rpa_get_device_error(None) == 0


def test_noalloc_bad_page_id_is_reported_in_the_scratch():
    b = workloads.decode_batch(seed=12, num_seqs=8, pool_pages=160)
    db = binding.Batch(b)
    plan = db.plan()
    assert binding.rpa_get_device_error(None) == 0
    pt = db.page_table.clone()
    pt[3, 0] = b.num_pages + 7            # outside the pool: the kernel skips it
    noalloc(db, b, plan, torch.empty_like(db.out), page_table=pt)
    assert binding.rpa_get_device_error(None) == binding.RPA_DEVERR_PAGE_ID
    # The read cleared the word; a good call leaves it clear and is right.
    got = noalloc(db, b, plan, torch.full_like(db.out, float("nan")))
    assert binding.rpa_get_device_error(None) == 0
    ref = oracle.attention(b.q, b.k_pages, b.v_pages, b.page_table, b.cu_q_lens, b.kv_lens,
                           b.window, b.sm_scale, precision=32)
    close(got, ref, "after a bad call")


def test_noalloc_rejects_prefill_and_oversized_plans():
    b = workloads.make_batch([1, 5], [40, 9], num_q_heads=8, num_kv_heads=1, head_dim=256,
                             page_size=128, seed=2)
    db = binding.Batch(b)
    plan = db.plan()
    with pytest.raises(binding.RpaError) as e:
        binding.rpa_forward_decode_noalloc(db.q, db.k_pages, db.v_pages, db.page_table,
                                           db.cu_q_lens, db.kv_lens, db.window, b.sm_scale,
                                           db.out, plan)
    assert e.value.status == binding.RPA_ERR_UNSUPPORTED
    # A plan needing more scratch than the fixed array is refused before any
    # pointer is used (so placeholder pointers are safe here).
    big = workloads.decode_batch(seed=3, num_seqs=512, lo=4096, hi=4096, pool_pages=16384,
                                 meta_only=True)
    plan_big = binding.rpa_plan(big.cu_q_lens, big.kv_lens, None, 8, 1, 256, 128,
                                big.max_pages_per_seq, big.num_pages, kv_split=64)
    assert plan_big.workspace_bytes > (32 << 20)
    fake = ctypes.c_void_p(1 << 20)
    st = binding.lib().rpa_forward_decode_noalloc(
        fake, fake, fake, fake, fake, fake, big.num_seqs, 8, 1, 256, 128, None, 0.0625, fake,
        None, plan_big.handle)
    assert st == binding.RPA_ERR_WORKSPACE_TOO_SMALL
