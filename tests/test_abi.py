"""The C ABI without a GPU: the library loads, exports what include/rpa.h
declares, and its host-side checks and scheduler behave as documented."""

from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

from ragged_paged_attention_rpa_gb300 import binding, build, workloads
from ragged_paged_attention_rpa_gb300.binding import (RPA_DTYPE_BF16, RPA_DTYPE_F32,
                                                      RPA_PATH_SIMT, RPA_PATH_TC, RpaError)

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "rpa.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rpa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(binding.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    for st in range(-6, 1):
        assert binding.status_string(st).startswith("RPA_")
    assert "unknown" in binding.status_string(-99)


def plan_of(b, **kw):
    return binding.rpa_plan(b.cu_q_lens, b.kv_lens, b.window, b.num_q_heads,
                            b.num_kv_heads, b.head_dim, b.page_size, b.max_pages_per_seq,
                            b.num_pages, dtype=RPA_DTYPE_BF16 if b.dtype == "bf16"
                            else RPA_DTYPE_F32, num_sms=152, **kw)


def ceil_div(a, b):
    return -(-a // b)


def test_decode_plan_covers_every_key():
    b = workloads.decode_batch(seed=1, meta_only=True)
    p = plan_of(b)
    info = p.info()
    assert info["num_decode_seqs"] == 128 and info["num_prefill_seqs"] == 0
    assert info["path"] == RPA_PATH_TC
    split = info["kv_split"]
    assert split % 64 == 0 and split > 0
    nsplit = [ceil_div(int(L), split) for L in b.kv_lens]
    assert info["max_splits"] == max(nsplit)
    # Workspace: 256-byte header, fp32 partial O and LSE for every split slot,
    # one int32 arrival counter per (sequence, KV head).
    if info["max_splits"] > 1:
        rows = b.num_seqs * info["max_splits"] * b.num_q_heads
        want = (256 + ceil_div(rows * b.head_dim * 4, 256) * 256 + ceil_div(rows * 4, 256) * 256
                + ceil_div(b.num_seqs * b.num_kv_heads * 4, 256) * 256)
    else:
        want = 256
    assert info["workspace_bytes"] == p.workspace_bytes == want


def test_decode_split_respects_window():
    b = workloads.mixed_batch(seed=4, meta_only=True)
    info = plan_of(b, kv_split=256).info()
    assert info["kv_split"] == 256
    vis = []
    for s in range(b.num_seqs):
        if b.cu_q_lens[s + 1] - b.cu_q_lens[s] != 1:
            continue
        L, w = int(b.kv_lens[s]), int(b.window[s])
        vis.append(min(L, w) if w > 0 else L)
    assert info["max_splits"] == max(ceil_div(v, 256) for v in vis)
    assert info["num_decode_seqs"] == 512 and info["num_prefill_seqs"] == 4


def test_forced_split_is_rounded_to_64():
    b = workloads.decode_batch(seed=1, meta_only=True)
    assert plan_of(b, kv_split=100).info()["kv_split"] == 128


def test_split_count_is_capped():
    # 64 splits at most per sequence: a 64-token split of a 100k-token context
    # is raised to ceil(100000 / 64) rounded up to 64.
    b = workloads.make_batch([1], [100000], num_q_heads=8, num_kv_heads=1, head_dim=256,
                             page_size=128, meta_only=True)
    info = plan_of(b, kv_split=64).info()
    assert info["max_splits"] <= 64 and info["kv_split"] == 1600


def test_f32_takes_the_simt_path():
    b = workloads.make_batch([3, 1], [9, 5], num_q_heads=4, num_kv_heads=2, head_dim=64,
                             page_size=16, dtype="f32", seed=3)
    assert plan_of(b).info()["path"] == RPA_PATH_SIMT
    with pytest.raises(RpaError) as e:
        plan_of(b, path=RPA_PATH_TC)
    assert e.value.status == binding.RPA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), binding.RPA_ERR_UNSUPPORTED),
    (dict(page_size=24), binding.RPA_ERR_UNSUPPORTED),
    (dict(num_kv_heads=3), binding.RPA_ERR_INVALID_ARG),
    (dict(max_pages_per_seq=1), binding.RPA_ERR_INVALID_ARG),
])
def test_plan_rejects(kw, status):
    b = workloads.make_batch([3, 1], [40, 5], num_q_heads=4, num_kv_heads=2, head_dim=64,
                             page_size=16, seed=3)
    args = dict(num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16,
                max_pages_per_seq=b.max_pages_per_seq, num_pages=b.num_pages)
    args.update(kw)
    with pytest.raises(RpaError) as e:
        binding.rpa_plan(b.cu_q_lens, b.kv_lens, None, **args)
    assert e.value.status == status


def test_plan_rejects_bad_lengths():
    with pytest.raises(RpaError) as e:
        binding.rpa_plan([0, 5], [4], None, 4, 1, 64, 16, 1, 1)    # q_len > kv_len
    assert e.value.status == binding.RPA_ERR_INVALID_ARG
    with pytest.raises(RpaError):
        binding.rpa_plan([1, 5], [9], None, 4, 1, 64, 16, 1, 1)    # cu_q_lens[0] != 0


def test_empty_batch_plans():
    p = binding.rpa_plan([0], np.zeros(0, np.int32), None, 8, 1, 256, 128, 1, 1)
    info = p.info()
    assert info["num_decode_seqs"] == 0 and info["workspace_bytes"] == 256


def test_forward_checks_before_any_launch():
    """Host-side argument checks return before anything is enqueued (no GPU)."""
    b = workloads.decode_batch(seed=1, num_seqs=4, meta_only=True)
    p = plan_of(b)
    L = binding.lib()
    fake = ctypes.c_void_p(1 << 20)      # never dereferenced: checks fail first
    ws = ctypes.c_void_p(1 << 21)
    args = [fake] * 6 + [b.num_seqs, 8, 1, 256, 128, None, 0.0625, fake, None, p.handle,
                         ws, p.workspace_bytes]
    bad = list(args)
    bad[7] = 16                                           # num_q_heads differs
    assert L.rpa_forward(*bad) == binding.RPA_ERR_PLAN_MISMATCH
    bad = list(args)
    bad[11] = fake                                        # window given, plan had none
    assert L.rpa_forward(*bad) == binding.RPA_ERR_PLAN_MISMATCH
    bad = list(args)
    bad[17] = p.workspace_bytes - 1
    if p.workspace_bytes > 256:
        assert L.rpa_forward(*bad) == binding.RPA_ERR_WORKSPACE_TOO_SMALL
    bad = list(args)
    bad[16] = ctypes.c_void_p((1 << 21) + 8)              # workspace not 256-B aligned
    assert L.rpa_forward(*bad) == binding.RPA_ERR_INVALID_ARG
    bad = list(args)
    bad[0] = None                                         # null q
    assert L.rpa_forward(*bad) == binding.RPA_ERR_INVALID_ARG
    bad = list(args)
    bad[1] = ctypes.c_void_p((1 << 20) + 64)              # k_pages not 128-B aligned
    assert L.rpa_forward(*bad) == binding.RPA_ERR_INVALID_ARG
