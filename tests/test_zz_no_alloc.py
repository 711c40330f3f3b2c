"""rpa_forward_decode_noalloc: decode for callers that cannot allocate device
memory at call time (their memory is owned by another allocator, or a
real-time loop must not call cudaMalloc).  It runs the same split-KV decode
kernel as rpa_forward but keeps its scratch in a fixed array inside librpa.

Checked through the C ABI against rpa_forward with a caller workspace, on two
calls in a row (the second call must not see stale counters or partials from
the first).  This file sorts last so that a failure here stops a -x run only
after every other test has run; it also passes alone in a fresh process.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from ragged_paged_attention_rpa_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def test_noalloc_decode_matches_rpa_forward_twice():
    b = workloads.decode_batch(seed=11, num_seqs=96, pool_pages=1600)
    db = binding.Batch(b)
    plan = db.plan(kv_split=256)          # several splits per sequence: uses the scratch
    info = plan.info()
    assert info["max_splits"] > 1 and plan.workspace_bytes <= (32 << 20)
    ws = binding.alloc_workspace(plan)
    ref = db.forward(plan, ws).float().cpu().numpy()
    assert binding.rpa_get_device_error(ws) == 0
    for call in range(2):
        out = torch.full_like(db.out, float("nan"))
        binding.rpa_forward_decode_noalloc(db.q, db.k_pages, db.v_pages, db.page_table,
                                           db.cu_q_lens, db.kv_lens, db.window, b.sm_scale,
                                           out, plan)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all(), "call %d left outputs unwritten" % call
        e = np.abs(got - ref)
        assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN, (call, e.max(), e.mean())


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
