"""rpa_forward captured into a CUDA graph: the call only enqueues kernel
launches, so a capture on the caller's stream replays the same attention.
The replayed output must equal the oracle's within the bf16 tolerance and the
direct call's output bit for bit (same kernels, same schedule); trace marks
taken during the capture become graph nodes whose times are read after the
replay."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from ragged_paged_attention_rpa_gb300 import binding, build, workloads

from .test_gpu_parity import assert_bf16_close, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def small_mixed(seed):
    # Decode rows long enough to be cut across CTAs (combine kernel), two
    # prefill sequences with windows (prefill kernel).
    ql = [1] * 24 + [96, 200]
    kv = [int(x) for x in np.random.default_rng(seed).integers(200, 6000, size=24)] + [300, 900]
    win = [0 if i % 2 else 256 for i in range(len(ql))]
    return workloads.make_batch(ql, kv, num_q_heads=8, num_kv_heads=1, head_dim=256,
                                page_size=128, windows=win, seed=seed, dtype="bf16")


@pytest.mark.parametrize("seed", [900, 901])
def test_graph_replay_matches_direct_call_and_oracle(seed):
    b = small_mixed(seed)
    db = binding.Batch(b)
    plan = db.plan()
    info = plan.info()
    assert info["num_prefill_seqs"] == 2
    ws = binding.alloc_workspace(plan)
    direct = db.forward(plan, ws).clone()
    assert binding.rpa_get_device_error(ws) == 0

    db.out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        db.call(plan, ws)()
    torch.cuda.synchronize()
    assert not db.out.any()            # capture ran nothing
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert binding.rpa_get_device_error(ws) == 0
    assert torch.equal(db.out.view(torch.int16), direct.view(torch.int16))
    got = db.out.float().cpu().numpy().reshape(-1, b.head_dim).astype(np.float64)
    assert_bf16_close(got, oracle_rows(b), "graph replay seed %d" % seed)


def test_trace_marks_inside_a_graph():
    b = small_mixed(902)
    db = binding.Batch(b)
    plan = db.plan()
    ws = binding.alloc_workspace(plan)
    db.forward(plan, ws)
    torch.cuda.synchronize()
    binding.rpa_trace_begin(64)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        db.call(plan, ws)()
    g.replay()
    torch.cuda.synchronize()
    recs = binding.rpa_trace_end(64)
    names = [n for n, _ in recs]
    assert "decode_split" in names and "prefill_tc" in names, names
    assert all(ms > 0.0 for _, ms in recs), recs
