"""GPU parity of the decode over fp8 (e4m3) K/V pages through the C ABI
(rpa_forward_fp8kv) against the oracle's attention over the dequantized
pages (code value times the KV head's scale)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ragged_paged_attention_rpa_gb300 import binding, workloads

from .test_gpu_parity import assert_bf16_close, unseen_slots

pytestmark = pytest.mark.gpu

CASES = [
    # (kv_lens, Hq, Hkv, D, P, windows)
    ([1, 2, 15, 16, 17, 127, 128, 129, 700], 8, 1, 256, 128, None),
    ([3, 64, 65, 200, 1000, 5, 40], 8, 2, 128, 32, [0, 16, 0, 100, 0, 2, 9]),
    ([2000, 37, 513, 90], 4, 2, 128, 16, [1000, 0, 64, 0]),
    ([129, 4097, 64, 1], 16, 2, 256, 64, None),
]


def fp8_oracle(b):
    return oracle.attention(oracle.bf16_bits_to_f32(b.q), oracle.dequantize_kv(b.k_fp8, b.k_scale),
                            oracle.dequantize_kv(b.v_fp8, b.v_scale), b.page_table, b.cu_q_lens,
                            b.kv_lens, b.window, b.sm_scale, precision=32)


def run_fp8(b):
    db = binding.Batch(b)
    plan = db.plan(kv_dtype=binding.RPA_DTYPE_FP8_E4M3)
    ws = binding.alloc_workspace(plan)
    k8 = torch.from_numpy(b.k_fp8).cuda()
    v8 = torch.from_numpy(b.v_fp8).cuda()
    ks = torch.from_numpy(b.k_scale).cuda()
    vs = torch.from_numpy(b.v_scale).cuda()
    db.out.fill_(float("nan"))
    binding.rpa_forward_fp8kv(db.q, k8, v8, ks, vs, db.page_table, db.cu_q_lens, db.kv_lens,
                              db.window, b.sm_scale, db.out, plan, ws)
    err = binding.rpa_get_device_error(ws)
    torch.cuda.synchronize()
    return db.out.float().cpu().numpy().reshape(-1, b.head_dim).astype(np.float64), err, plan


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fp8_decode_matches_oracle(case):
    kv, hq, hkv, d, p, win = CASES[case]
    b = workloads.with_fp8_kv(workloads.make_batch([1] * len(kv), kv, num_q_heads=hq,
                                                   num_kv_heads=hkv, head_dim=d, page_size=p,
                                                   windows=win, seed=800 + case))
    got, err, plan = run_fp8(b)
    assert err == 0 and plan.info()["kv_dtype"] == binding.RPA_DTYPE_FP8_E4M3
    assert_bf16_close(got, fp8_oracle(b), "fp8 decode case %d" % case)


def test_fp8_decode_workload():
    b = workloads.WORKLOADS["decode_fp8"]()
    got, err, _ = run_fp8(b)
    assert err == 0
    assert_bf16_close(got, fp8_oracle(b), "fp8 decode workload")


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fp8_decode_poisoned(case):
    """e4m3 NaN (S.1111.111) in every fp8 slot no query sees."""
    kv, hq, hkv, d, p, win = CASES[case]
    b = workloads.with_fp8_kv(workloads.make_batch([1] * len(kv), kv, num_q_heads=hq,
                                                   num_kv_heads=hkv, head_dim=d, page_size=p,
                                                   windows=win, pool_pages=sum(-(-x // p) for x in kv) + 3,
                                                   seed=870 + case))
    mask = unseen_slots(b)
    assert mask.any()
    k8, v8 = b.k_fp8.copy(), b.v_fp8.copy()
    k8[mask] = 0x7F
    v8[mask] = 0xFF
    b = workloads.Batch(**{**b.__dict__, "k_fp8": k8, "v_fp8": v8})
    got, err, _ = run_fp8(b)
    assert err == 0
    assert_bf16_close(got, fp8_oracle(b), "poisoned fp8 decode case %d" % case)


def test_bf16_entry_point_refuses_an_fp8_plan():
    b = workloads.with_fp8_kv(workloads.make_batch([1, 1], [40, 9], num_q_heads=8,
                                                   num_kv_heads=1, head_dim=128, page_size=16,
                                                   seed=850))
    db = binding.Batch(b)
    plan = db.plan(kv_dtype=binding.RPA_DTYPE_FP8_E4M3)
    ws = binding.alloc_workspace(plan)
    with pytest.raises(binding.RpaError) as e:
        db.forward(plan, ws)
    assert e.value.status == binding.RPA_ERR_PLAN_MISMATCH
