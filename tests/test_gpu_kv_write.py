"""GPU parity of the KV-cache write (rpa_write_kv) and of the write followed
by attention (rpa_forward_kv), through the C ABI: the pools the kernel
writes equal the oracle's bit for bit, and the attention over them equals the
oracle's attention over the batch's own pools."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ragged_paged_attention_rpa_gb300 import binding, workloads

from .test_gpu_parity import assert_bf16_close, oracle_rows

pytestmark = pytest.mark.gpu

CASES = [
    # (q_lens, kv_lens, Hq, Hkv, D, P, windows, dtype)
    ([1, 7, 1, 40], [33, 7, 200, 300], 8, 2, 64, 16, [0, 0, 5, 64], "bf16"),
    ([1] * 5 + [130], [129, 1, 700, 64, 17, 400], 8, 1, 256, 128, None, "bf16"),
    ([3, 1, 20], [9, 5, 40], 4, 2, 64, 16, [0, 3, 0], "f32"),
]


def new_rows(b):
    """The new tokens' K/V rows ([total_q, Hkv, D]) and the pools with their
    slots zeroed (the cache before the step)."""
    P = b.page_size
    kn = np.zeros((b.total_q,) + b.k_pages.shape[2:], dtype=b.k_pages.dtype)
    vn = np.zeros_like(kn)
    kz, vz = b.k_pages.copy(), b.v_pages.copy()
    for s in range(b.num_seqs):
        ql = int(b.cu_q_lens[s + 1] - b.cu_q_lens[s])
        L = int(b.kv_lens[s])
        for i in range(ql):
            t, pos = int(b.cu_q_lens[s]) + i, L - ql + i
            page = int(b.page_table[s, pos // P])
            kn[t], vn[t] = b.k_pages[page, pos % P], b.v_pages[page, pos % P]
            kz[page, pos % P] = 0
            vz[page, pos % P] = 0
    return kn, vn, kz, vz


def dev(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.cuda()


def host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


@pytest.mark.parametrize("case", range(len(CASES)))
def test_write_kv_matches_oracle_bitwise(case):
    ql, kv, hq, hkv, d, p, win, dtype = CASES[case]
    b = workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=p, windows=win, seed=700 + case, dtype=dtype)
    kn, vn, kz, vz = new_rows(b)
    want_k, want_v = oracle.write_kv(kz, vz, kn, vn, b.page_table, b.cu_q_lens, b.kv_lens)
    kp, vp = dev(kz, dtype), dev(vz, dtype)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    binding.rpa_write_kv(dev(kn, dtype), dev(vn, dtype), kp, vp, dev(b.page_table, "i32"),
                         dev(b.cu_q_lens, "i32"), dev(b.kv_lens, "i32"), b.num_pages,
                         workspace=ws)
    assert binding.rpa_get_device_error(ws) == 0
    assert np.array_equal(host(kp), want_k) and np.array_equal(host(vp), want_v)
    # The oracle's write restores the batch's own pools.
    assert np.array_equal(want_k, b.k_pages) and np.array_equal(want_v, b.v_pages)


@pytest.mark.parametrize("case", [0, 1])
def test_forward_kv_matches_oracle(case):
    ql, kv, hq, hkv, d, p, win, dtype = CASES[case]
    b = workloads.make_batch(ql, kv, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=p, windows=win, seed=710 + case, dtype=dtype)
    kn, vn, kz, vz = new_rows(b)
    db = binding.Batch(b)
    db.k_pages.copy_(dev(kz, dtype))
    db.v_pages.copy_(dev(vz, dtype))
    plan = db.plan()
    ws = binding.alloc_workspace(plan)
    binding.rpa_forward_kv(db.q, dev(kn, dtype), dev(vn, dtype), db.k_pages, db.v_pages,
                           db.page_table, db.cu_q_lens, db.kv_lens, db.window, b.sm_scale,
                           db.out, plan, ws)
    assert binding.rpa_get_device_error(ws) == 0
    torch.cuda.synchronize()
    assert np.array_equal(host(db.k_pages), b.k_pages)
    got = db.out.float().cpu().numpy().reshape(-1, d).astype(np.float64)
    assert_bf16_close(got, oracle_rows(b), "forward_kv case %d" % case)


def test_write_kv_reports_a_bad_page():
    b = workloads.make_batch([2], [10], num_q_heads=2, num_kv_heads=1, head_dim=64,
                             page_size=16, seed=720)
    kn, vn, kz, vz = new_rows(b)
    pt = b.page_table.copy()
    pt[0, 0] = b.num_pages + 5          # the new tokens' page: out of range
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    kp = dev(kz, "bf16")
    binding.rpa_write_kv(dev(kn, "bf16"), dev(vn, "bf16"), kp, dev(vz, "bf16"), dev(pt, "i32"),
                         dev(b.cu_q_lens, "i32"), dev(b.kv_lens, "i32"), b.num_pages,
                         workspace=ws)
    assert binding.rpa_get_device_error(ws) == binding.RPA_DEVERR_PAGE_ID
    assert np.array_equal(host(kp), kz)   # nothing written
