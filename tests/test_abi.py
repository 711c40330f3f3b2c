"""The C ABI without a GPU: the library loads, exports what include/rpa.h
declares, and its host-side checks and scheduler behave as documented."""

from __future__ import annotations

import ctypes
import os
import re
import subprocess

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
    return sorted(set(re.findall(r"\b(rpa_[a-z0-9_]+)\s*\(", text)))


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


SEG_COST = 7  # blocks charged per segment a decode CTA's range touches


def decode_partition(b, num_sms=152, tokens_per_cta=0):
    """Expected decode schedule, restated from its definition: the 16-key
    blocks (on absolute 16-key boundaries) covering the visible keys of every
    (decode sequence, KV head), laid end to end and cut into contiguous
    ranges.  Forced: ranges of equal block counts.  Otherwise a range costs
    its blocks plus SEG_COST per segment it touches, and the cut takes the
    smallest cost cap T for which ranges grown as long as T allows number at
    most one per SM."""
    nb = []
    for s in range(b.num_seqs):
        if b.cu_q_lens[s + 1] - b.cu_q_lens[s] != 1:
            continue
        L = int(b.kv_lens[s])
        w = 0 if b.window is None else int(b.window[s])
        lo = max(0, L - w) if w > 0 else 0
        nb += [ceil_div(L, 16) - lo // 16] * b.num_kv_heads
    total = sum(nb)
    starts = np.concatenate([[0], np.cumsum(nb)]).astype(np.int64)

    def ranges_for(T):
        out, pos = [0], 0
        while pos < total:
            cost, end = 0, pos
            while end < total:
                k = int(np.searchsorted(starts, end, side="right")) - 1
                room = T - cost - SEG_COST
                if room <= 0 and end > pos:
                    break
                take = min(int(starts[k + 1]) - end, max(room, 1))
                cost += SEG_COST + take
                end += take
                if end < starts[k + 1]:
                    break
            out.append(end)
            pos = end
        return out

    if tokens_per_cta:
        bpc = ceil_div(tokens_per_cta, 16)
        bounds = list(range(0, total, bpc)) + [total]
    else:
        lo_T, hi_T = SEG_COST + 1, total + SEG_COST * (len(nb) + 1)
        while lo_T < hi_T:
            mid = (lo_T + hi_T) // 2
            if len(ranges_for(mid)) - 1 <= num_sms:
                hi_T = mid
            else:
                lo_T = mid + 1
        bounds = ranges_for(lo_T)
    n_ctas = len(bounds) - 1
    longest = max(bounds[i + 1] - bounds[i] for i in range(n_ctas))
    cta = lambda x: int(np.searchsorted(bounds, x, side="right")) - 1
    spans = [cta(starts[i + 1] - 1) - cta(starts[i]) + 1 for i in range(len(nb)) if nb[i] > 0]
    # The shared-memory table limits (64 segments, 512 pages per range) do
    # not bind for the batches these tests use.
    for i in range(n_ctas):
        assert sum(1 for k in range(len(nb))
                   if starts[k] < bounds[i + 1] and starts[k + 1] > bounds[i]) <= 64
    return dict(segments=len(nb), longest=longest, n_ctas=n_ctas, max_splits=max(spans))


def test_decode_plan_is_one_balanced_wave():
    b = workloads.decode_batch(seed=1, meta_only=True)
    p = plan_of(b)
    info = p.info()
    assert info["num_decode_seqs"] == 128 and info["num_prefill_seqs"] == 0
    assert info["path"] == RPA_PATH_TC
    want = decode_partition(b)
    assert info["kv_split"] == 16 * want["longest"]
    assert info["max_splits"] == want["max_splits"]
    assert want["n_ctas"] <= 152
    # Workspace: 256-byte header, two fp32 partial slots (G x D, plus G
    # log2-sum-exps) per decode CTA.
    G = b.num_q_heads // b.num_kv_heads
    slots = 2 * want["n_ctas"]
    want_ws = (256 + ceil_div(slots * G * b.head_dim * 4, 256) * 256
               + ceil_div(slots * G * 4, 256) * 256)
    assert info["workspace_bytes"] == p.workspace_bytes == want_ws


def test_decode_plan_respects_window_and_forced_range():
    b = workloads.mixed_batch(seed=4, meta_only=True)
    info = plan_of(b, kv_split=256).info()
    want = decode_partition(b, tokens_per_cta=256)
    assert info["kv_split"] == 256
    assert info["max_splits"] == want["max_splits"]
    assert info["num_decode_seqs"] == 512 and info["num_prefill_seqs"] == 4


def test_forced_range_is_rounded_to_16():
    b = workloads.decode_batch(seed=1, meta_only=True)
    assert plan_of(b, kv_split=100).info()["kv_split"] == 112


def test_cta_ranges_shrink_to_fit_the_page_table():
    # Page size 1: a 4096-token range would touch 4096 pages, more than a CTA's
    # shared-memory page table holds (512), so ranges shrink below 512 tokens.
    b = workloads.make_batch([1] * 152, [4096] * 152, num_q_heads=8, num_kv_heads=1,
                             head_dim=256, page_size=1, meta_only=True)
    info = plan_of(b).info()
    assert info["kv_split"] <= 512


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


def test_fp8_kv_plans_are_decode_only():
    b = workloads.make_batch([1, 1, 1], [40, 900, 7], num_q_heads=8, num_kv_heads=1,
                             head_dim=256, page_size=128, meta_only=True)
    info = plan_of(b, kv_dtype=binding.RPA_DTYPE_FP8_E4M3).info()
    assert info["kv_dtype"] == binding.RPA_DTYPE_FP8_E4M3 and info["path"] == RPA_PATH_TC
    assert plan_of(b).info()["kv_dtype"] == binding.RPA_DTYPE_BF16
    mixed = workloads.make_batch([1, 5], [40, 9], num_q_heads=8, num_kv_heads=1,
                                 head_dim=256, page_size=128, meta_only=True)
    with pytest.raises(RpaError) as e:
        plan_of(mixed, kv_dtype=binding.RPA_DTYPE_FP8_E4M3)
    assert e.value.status == binding.RPA_ERR_UNSUPPORTED
    d64 = workloads.make_batch([1, 1], [40, 9], num_q_heads=8, num_kv_heads=1, head_dim=64,
                               page_size=16, meta_only=True)
    with pytest.raises(RpaError) as e:
        plan_of(d64, kv_dtype=binding.RPA_DTYPE_FP8_E4M3)
    assert e.value.status == binding.RPA_ERR_UNSUPPORTED


def prefill_items(b, q_block):
    """(keys streamed, key tiles) of every prefill work item (sequence, query
    block): the keys from the first visible key of its first query to its last
    query's position; the 128-key tiles starting on a multiple of 64 at or
    below that first key.  Restated from the attention's visibility rule."""
    items = []
    for s in range(b.num_seqs):
        ql = int(b.cu_q_lens[s + 1] - b.cu_q_lens[s])
        if ql <= 1:
            continue
        L = int(b.kv_lens[s])
        w = 0 if b.window is None else int(b.window[s])
        for blk in range(-(-ql // q_block)):
            pos0 = L - ql + blk * q_block
            pos1 = min(L - ql + (blk + 1) * q_block, L) - 1
            lo = pos0 - (w - 1) if (w > 0 and pos0 - (w - 1) > 0) else 0
            items.append((pos1 - lo + 1, (pos1 - lo // 64 * 64) // 128 + 1))
    return items


def prefill_tiles(b, q_block):
    """Key tiles (128 keys, starting on a multiple of 64 at or below the first
    visible key) of every prefill work item (sequence, query block), restated
    from the attention's visibility rule."""
    tiles = []
    for s in range(b.num_seqs):
        ql = int(b.cu_q_lens[s + 1] - b.cu_q_lens[s])
        if ql <= 1:
            continue
        L = int(b.kv_lens[s])
        w = 0 if b.window is None else int(b.window[s])
        for blk in range(-(-ql // q_block)):
            pos0 = L - ql + blk * q_block
            pos1 = min(L - ql + (blk + 1) * q_block, L) - 1
            lo = pos0 - (w - 1) if (w > 0 and pos0 - (w - 1) > 0) else 0
            tiles.append((pos1 - lo // 64 * 64) // 128 + 1)
    return tiles


def range_parts(tiles, per):
    """Items' tiles laid end to end and cut into ranges of `per` tiles: the
    ranges, and the parts of items that cross a range boundary (and the items
    that do not)."""
    parts, whole, pos = 0, 0, 0
    for t in tiles:
        first, last = pos // per, (pos + t - 1) // per
        if last > first:
            parts += last - first + 1
        else:
            whole += 1
        pos += t
    return -(-pos // per), parts, whole


def test_prefill_items_split_on_request():
    """prefill_split = n lays the items' key tiles end to end (sequence order)
    and cuts them into one range of n tiles per CTA; items crossing a range
    boundary become parts.  Without the option nothing is split."""
    b = workloads.WORKLOADS["spec_decode"](meta_only=True)
    assert plan_of(b).info()["prefill_split_items"] == 0
    per = 8
    info = plan_of(b, prefill_split=per).info()
    tiles = prefill_tiles(b, info["q_block"])           # sequence order
    grid, parts, whole = range_parts(tiles, per)
    assert info["prefill_ctas"] == grid
    assert info["prefill_split_parts"] == parts > 0
    assert info["num_prefill_items"] == parts + whole   # per-CTA lists, no padding
    # Workspace: one 128-row fp32 partial (and log2-sum-exps) per part.
    assert info["workspace_bytes"] >= parts * 128 * (256 + 1) * 4
    assert plan_of(b, prefill_split=-1).info()["prefill_split_items"] == 0


def test_prefill_split_forced():
    b = workloads.make_batch([300, 20], [4000, 900], num_q_heads=8, num_kv_heads=2,
                             head_dim=128, page_size=64, meta_only=True)
    info = plan_of(b, prefill_split=3).info()
    tiles = [t for t in prefill_tiles(b, info["q_block"]) for _ in range(2)]   # 2 KV heads
    grid, parts, _ = range_parts(tiles, 3)
    assert info["prefill_split_parts"] == parts and info["prefill_ctas"] == grid


def lpt_busiest(tiles, n, keys=None):
    """Longest processing time first: each item, longest first (by keys
    streamed when given, ties in list order), to the CTA with the fewest tiles
    so far (ties: lowest index); the busiest CTA's tiles."""
    import heapq
    order = range(len(tiles))
    if keys is not None:
        order = sorted(order, key=lambda i: (-keys[i], i))
    else:
        order = sorted(order, key=lambda i: (-tiles[i], i))
    heap = [(0, c) for c in range(n)]
    for i in order:
        load, c = heapq.heappop(heap)
        heapq.heappush(heap, (load + tiles[i], c))
    return max(load for load, _ in heap)


@pytest.mark.parametrize("name", ["causal_prefill", "swa_prefill", "mixed"])
def test_prefill_items_scheduled_longest_first_to_least_loaded(name):
    b = workloads.WORKLOADS[name](meta_only=True)
    info = plan_of(b).info()
    items = [it for it in prefill_items(b, info["q_block"]) for _ in range(b.num_kv_heads)]
    tiles = [t for _, t in items]
    n = min(len(tiles), info["prefill_sms"] or 152)
    assert info["prefill_ctas"] == n
    assert info["prefill_max_tiles"] == lpt_busiest(tiles, n, keys=[k for k, _ in items])
    # Striding the longest-first list would load the busiest CTA more.
    by_len = sorted(tiles, reverse=True)
    assert max(sum(by_len[c::n]) for c in range(n)) >= info["prefill_max_tiles"]


def test_new_token_entry_points_check_before_any_launch():
    """rpa_write_kv, rpa_qkv_prologue and rpa_forward_qkv reject bad arguments
    on the host, before anything is enqueued (no GPU)."""
    b = workloads.decode_batch(seed=1, num_seqs=4, meta_only=True)
    p = plan_of(b)
    L = binding.lib()
    fake = ctypes.c_void_p(1 << 20)
    ws = ctypes.c_void_p(1 << 21)
    w = ctypes.c_void_p(1 << 22)
    norm = binding.QkvNorm(w.value, w.value, None, 1e-6, 10000.0)
    # rpa_write_kv: page_size not a power of two; head_dim * 2 B not a multiple of 16 B.
    kv_args = [fake] * 7 + [4, 4, 1, 256, 128, 16, 4096, binding.RPA_DTYPE_BF16, None, None]
    bad = list(kv_args)
    bad[11] = 96
    assert L.rpa_write_kv(*bad) == binding.RPA_ERR_INVALID_ARG
    bad = list(kv_args)
    bad[10] = 4
    assert L.rpa_write_kv(*bad) == binding.RPA_ERR_UNSUPPORTED
    # rpa_qkv_prologue: unsupported head_dim, misaligned q, negative eps, null norm.
    pro = [fake, fake, fake, ctypes.byref(norm), fake, fake, fake, fake, fake, fake,
           4, 4, 8, 1, 256, 128, 16, 4096, binding.RPA_DTYPE_BF16, None, None]
    bad = list(pro)
    bad[14] = 96
    assert L.rpa_qkv_prologue(*bad) == binding.RPA_ERR_UNSUPPORTED
    bad = list(pro)
    bad[0] = ctypes.c_void_p((1 << 20) + 8)
    assert L.rpa_qkv_prologue(*bad) == binding.RPA_ERR_INVALID_ARG
    neg = binding.QkvNorm(w.value, w.value, None, -1.0, 10000.0)
    bad = list(pro)
    bad[3] = ctypes.byref(neg)
    assert L.rpa_qkv_prologue(*bad) == binding.RPA_ERR_INVALID_ARG
    bad = list(pro)
    bad[3] = None
    assert L.rpa_qkv_prologue(*bad) == binding.RPA_ERR_INVALID_ARG
    # rpa_forward_qkv: the plan's scalars must match; workspace size and alignment.
    fq = [fake, fake, fake, ctypes.byref(norm), fake, fake, fake, fake, fake, fake,
          b.num_seqs, 8, 1, 256, 128, None, 0.0625, fake, None, p.handle, ws, p.workspace_bytes]
    bad = list(fq)
    bad[11] = 16
    assert L.rpa_forward_qkv(*bad) == binding.RPA_ERR_PLAN_MISMATCH
    bad = list(fq)
    bad[20] = ctypes.c_void_p((1 << 21) + 8)
    assert L.rpa_forward_qkv(*bad) == binding.RPA_ERR_INVALID_ARG
    bad = list(fq)
    bad[4] = None                                         # null q_buf
    assert L.rpa_forward_qkv(*bad) == binding.RPA_ERR_INVALID_ARG


def test_plan_rejects_bad_split_option():
    b = workloads.decode_batch(seed=1, num_seqs=4, meta_only=True)
    with pytest.raises(binding.RpaError):
        plan_of(b, prefill_split=-2)


def test_prefill_lists_fall_back_to_striding_beyond_one_launch():
    """More items than one launch carries (sliding-window 8k with 16-token
    query blocks: 8192 items): the items stay longest first and CTA c takes
    c, c + 152, ...; the busiest CTA's tiles follow that striding."""
    b = workloads.WORKLOADS["swa_prefill"](meta_only=True)
    info = plan_of(b, q_block=16).info()
    tiles = sorted((t for t in prefill_tiles(b, 16) for _ in range(b.num_kv_heads)), reverse=True)
    assert info["num_prefill_items"] == len(tiles) == 8192
    assert info["prefill_max_tiles"] == max(sum(tiles[c::152]) for c in range(152))


def test_decode_plan_splits_into_launches_by_segment_count():
    """Thousands of decode sequences exceed one launch's segment table: the
    plan issues several launches, every block still covered exactly once."""
    rng = np.random.default_rng(5)
    n = 2500
    kv = rng.integers(1, 65, size=n).tolist()
    b = workloads.make_batch([1] * n, kv, num_q_heads=8, num_kv_heads=2, head_dim=128,
                             page_size=16, meta_only=True)
    info = plan_of(b).info()
    assert info["num_decode_seqs"] == n and info["path"] == binding.RPA_PATH_TC
    # Workspace holds two partial slots per decode CTA of every launch.
    assert info["workspace_bytes"] > 256


def test_header_is_plain_c(tmp_path):
    """include/rpa.h compiles as C11 and librpa links and plans from C."""
    exe = str(tmp_path / "abi_c_check")
    src = os.path.join(os.path.dirname(__file__), "csrc", "abi_c_check.c")
    lib_dir = os.path.dirname(binding.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I" + build.INCLUDE, src, "-o", exe,
                    "-L" + lib_dir, "-lrpa", "-Wl,-rpath," + lib_dir], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("c abi ok")


@pytest.mark.parametrize("seed", range(12))
def test_decode_plan_matches_restatement_on_random_batches(seed):
    """Random decode batches (sequence counts, lengths, windows, KV heads,
    page sizes): the plan's longest range, most-split sequence and CTA count
    (through the workspace size) equal the restated cost-balanced cut."""
    rng = np.random.default_rng(4000 + seed)
    hkv = int(rng.choice([1, 2, 4]))
    n = int(rng.integers(1, 1024 // hkv + 1))    # one launch: at most 1024 segments
    P = int(rng.choice([16, 32, 64, 128]))
    # Lengths whose ranges stay within the kernel's page table (512 pages per
    # range), which the restatement does not model.
    kv = rng.integers(1, int(rng.choice([64, 600] if P < 64 else [64, 600, 4000])) + 1,
                      size=n).tolist()
    win = [int(w) if rng.random() < 0.4 else 0 for w in rng.integers(1, 2000, size=n)]
    b = workloads.make_batch([1] * n, kv, num_q_heads=8 * hkv, num_kv_heads=hkv, head_dim=128,
                             page_size=P, windows=win, meta_only=True)
    info = plan_of(b).info()
    want = decode_partition(b)
    assert info["kv_split"] == 16 * want["longest"]
    assert info["max_splits"] == want["max_splits"]
    G = b.num_q_heads // b.num_kv_heads
    slots = 2 * want["n_ctas"]
    assert info["workspace_bytes"] == (256 + ceil_div(slots * G * 128 * 4, 256) * 256
                                       + ceil_div(slots * G * 4, 256) * 256)


def test_decode_plan_falls_back_to_fixed_ranges_when_tables_bind():
    """1000 sequences of 4000 keys on 16-token pages: one range per SM would
    touch ~1650 pages, more than a CTA's page table holds (512), so no cut
    into 152 ranges is feasible; the plan takes fixed ranges small enough for
    the table, in several waves, covering every block."""
    b = workloads.make_batch([1] * 1000, [4000] * 1000, num_q_heads=8, num_kv_heads=1,
                             head_dim=128, page_size=16, meta_only=True)
    info = plan_of(b).info()
    bpc = info["kv_split"] // 16
    total = 1000 * ceil_div(4000, 16)
    n_ctas = ceil_div(total, bpc)
    assert n_ctas > 152 and bpc <= 512
    slots = 2 * n_ctas
    assert info["workspace_bytes"] == (256 + ceil_div(slots * 8 * 128 * 4, 256) * 256
                                       + ceil_div(slots * 8 * 4, 256) * 256)


@pytest.mark.parametrize("seed", range(10))
def test_prefill_schedule_matches_restatement_on_random_batches(seed):
    rng = np.random.default_rng(5000 + seed)
    n = int(rng.integers(1, 12))
    hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8]))
    ql = rng.integers(2, 1500, size=n)
    kv = (ql + rng.integers(0, 3000, size=n)).tolist()
    win = [int(w) if rng.random() < 0.5 else 0 for w in rng.integers(1, 2000, size=n)]
    b = workloads.make_batch(ql.tolist(), kv, num_q_heads=G * hkv, num_kv_heads=hkv,
                             head_dim=128, page_size=64, windows=win, meta_only=True)
    info = plan_of(b).info()
    items = [it for it in prefill_items(b, info["q_block"]) for _ in range(hkv)]
    if len(items) > 2048:      # beyond one launch: striding (tested separately)
        pytest.skip("more items than one launch carries")
    n_ctas = min(len(items), 152)
    assert info["prefill_ctas"] == n_ctas
    assert info["prefill_max_tiles"] == lpt_busiest([t for _, t in items], n_ctas,
                                                    keys=[k for k, _ in items])


def test_plan_log_line_when_asked():
    """RPA_LOG=1: every rpa_plan prints one line about the plan to stderr."""
    code = ("import sys; sys.path.insert(0, %r)\n"
            "from ragged_paged_attention_rpa_gb300 import binding, workloads\n"
            "b = workloads.decode_batch(seed=1, meta_only=True)\n"
            "binding.rpa_plan(b.cu_q_lens, b.kv_lens, b.window, 8, 1, 256, 128,\n"
            "                 b.max_pages_per_seq, b.num_pages, num_sms=152)\n" % build.ROOT)
    import sys as _sys
    on = subprocess.run([_sys.executable, "-c", code], capture_output=True, text=True,
                        env=dict(os.environ, RPA_LOG="1"), timeout=120)
    off = subprocess.run([_sys.executable, "-c", code], capture_output=True, text=True,
                         env={k: v for k, v in os.environ.items() if k != "RPA_LOG"}, timeout=120)
    assert on.returncode == 0 and off.returncode == 0, on.stderr + off.stderr
    assert on.stderr.count("librpa plan: 128 seqs (128 decode, 0 prefill)") == 1, on.stderr
    assert "librpa plan" not in off.stderr


def test_q_block_is_honoured_or_refused():
    """A requested prefill query block is used as asked: up to one 128-row
    tile per CTA (128 / G tokens; G = 2 here, so 64), twice that on SM pairs
    (half per SM), and anything larger is refused, never silently shrunk."""
    b = workloads.WORKLOADS["swa_prefill"](meta_only=True)
    for qb in (8, 16, 32, 64):
        info = plan_of(b, q_block=qb).info()
        assert info["q_block"] == qb and info["prefill_pairs"] == 0
    info = plan_of(b, q_block=128).info()
    assert info["q_block"] == 128 and info["prefill_pairs"] == 1
    assert info["num_prefill_items"] == b.num_kv_heads * 8192 // 128
    info = plan_of(b, q_block=64, prefill_pairs=2).info()
    assert info["q_block"] == 64 and info["prefill_pairs"] == 1
    for qb in (256, 512, 129, 96 + 1):
        with pytest.raises(RpaError) as e:
            plan_of(b, q_block=qb)
        assert e.value.status == binding.RPA_ERR_UNSUPPORTED, qb
    # Multi-token decode at G = 8: one tile holds 16 tokens, a pair 32.
    s = workloads.spec_decode_batch(meta_only=True)
    assert plan_of(s, q_block=16).info()["q_block"] == 16
    assert plan_of(s, q_block=32).info()["prefill_pairs"] == 1
    with pytest.raises(RpaError):
        plan_of(s, q_block=64)


# The planner's cost model of a mixed batch's two grids, restated: decode
# streams its visible 16-key blocks' K and V at up to 78 GB/s per SM until
# 5000 GB/s, plus 8 us; the prefill takes 1.6 us per key tile and 3.2 us per
# item epilogue at D = 256 (scaled by D / 256), plus 20 us, its tiles per CTA
# at least those of the longest item.
def mixed_costs(b, n_sms=152):
    ql = np.diff(b.cu_q_lens)
    dec_bytes = 0.0
    for s in np.where(ql == 1)[0]:
        L = int(b.kv_lens[s])
        w = 0 if b.window is None else int(b.window[s])
        lo = L - w if (w > 0 and L - w > 0) else 0
        dec_bytes += (ceil_div(L, 16) - lo // 16) * 16 * b.num_kv_heads * b.head_dim * 4
    qb = 128 // (b.num_q_heads // b.num_kv_heads)
    tiles = [t for _, t in prefill_items(b, qb) for _ in range(b.num_kv_heads)]
    f = b.head_dim / 256

    def dec(x):
        return dec_bytes / min(x * 78.0, 5000.0) * 1e-3 + 8.0

    def pre(y):
        return (max(sum(tiles) / y, max(tiles)) * 1.6 * f + ceil_div(len(tiles), y) * 3.2 * f
                + 20.0)
    return dec, pre


def test_mixed_batch_grids_split_the_sms_by_the_cost_model():
    """A batch with decode and prefill sequences runs its two persistent grids
    side by side on disjoint SMs, split where the modelled times of the two
    are most even (the larger of the two smallest), when that beats running
    them one after the other; -1 keeps them sequential, n > 0 forces the
    split."""
    b = workloads.mixed_batch(seed=4, meta_only=True)
    dec, pre = mixed_costs(b)
    best = min(range(1, 152), key=lambda x: (max(dec(x), pre(152 - x)), x))
    assert max(dec(best), pre(152 - best)) < dec(152) + pre(152)
    info = plan_of(b).info()
    assert info["decode_sms"] == best and info["prefill_sms"] == 152 - best
    assert info["prefill_ctas"] == min(152 - best, info["num_prefill_items"])
    seq = plan_of(b, decode_sms=-1).info()
    assert seq["decode_sms"] == 0 and seq["prefill_sms"] == 0 and seq["prefill_ctas"] == 152
    forced = plan_of(b, decode_sms=100).info()
    assert forced["decode_sms"] == 100 and forced["prefill_sms"] == 52
    with pytest.raises(RpaError):
        plan_of(b, decode_sms=-2)
    # Decode-only and prefill-only batches have nothing to overlap.
    assert plan_of(workloads.decode_batch(meta_only=True)).info()["decode_sms"] == 0
    assert plan_of(workloads.WORKLOADS["swa_prefill"](meta_only=True)).info()["decode_sms"] == 0


def test_decode_kernel_option():
    """decode_kernel picks the split-KV decode kernel: 1 the CUDA-core one (any
    tensor-core decode shape, fp8 pages too), 2 the tensor-core one (bf16
    pages, head_dim 128 or 256, G <= 8, pages of >= 16 tokens) or
    RPA_ERR_UNSUPPORTED; 0 the planner's choice.  The plan reports which."""
    b = workloads.decode_batch(meta_only=True)
    assert plan_of(b, decode_kernel=1).info()["decode_kernel"] == 1
    assert plan_of(b, decode_kernel=2).info()["decode_kernel"] == 2
    assert plan_of(b).info()["decode_kernel"] in (1, 2)
    for bad in (-1, 3):
        with pytest.raises(RpaError) as e:
            plan_of(b, decode_kernel=bad)
        assert e.value.status == binding.RPA_ERR_INVALID_ARG
    with pytest.raises(RpaError) as e:
        plan_of(b, decode_kernel=2, kv_dtype=binding.RPA_DTYPE_FP8_E4M3)
    assert e.value.status == binding.RPA_ERR_UNSUPPORTED
    fp8 = plan_of(b, decode_kernel=1, kv_dtype=binding.RPA_DTYPE_FP8_E4M3).info()
    assert fp8["decode_kernel"] == 1
    d64 = workloads.make_batch([1, 1], [40, 9], num_q_heads=8, num_kv_heads=1, head_dim=64,
                               page_size=16, meta_only=True)
    with pytest.raises(RpaError) as e:
        plan_of(d64, decode_kernel=2)
    assert e.value.status == binding.RPA_ERR_UNSUPPORTED
    assert plan_of(d64).info()["decode_kernel"] == 1
    # No decode sequence: no decode kernel, whatever was asked.
    pre = workloads.WORKLOADS["swa_prefill"](meta_only=True)
    assert plan_of(pre, decode_kernel=2).info()["decode_kernel"] == 0
    # The CUDA-core (SIMT) path: no split-KV decode either.
    assert plan_of(b, path=binding.RPA_PATH_SIMT).info()["decode_kernel"] == 0


@pytest.mark.parametrize("name", ["causal_prefill", "swa_prefill", "mixed"])
def test_prefill_items_taken_dynamically_by_default(name):
    """Single-SM prefill items are taken longest first by whichever CTA gets
    free (prefill_dynamic = 0, the default); -1 keeps the planner's per-CTA
    lists.  Both plans hold the same items, grid and LPT makespan estimate."""
    b = workloads.WORKLOADS[name](meta_only=True)
    dyn = plan_of(b).info()
    fixed = plan_of(b, prefill_dynamic=-1).info()
    assert dyn["prefill_dynamic"] == 1 and fixed["prefill_dynamic"] == 0
    for k in ("num_prefill_items", "prefill_ctas", "prefill_max_tiles", "q_block"):
        assert dyn[k] == fixed[k], k
    for bad in (-2, 1):
        with pytest.raises(RpaError) as e:
            plan_of(b, prefill_dynamic=bad)
        assert e.value.status == binding.RPA_ERR_INVALID_ARG
    # Split items and SM pairs keep fixed lists (a split that does not fit
    # one launch falls back to whole items).
    sp = plan_of(b, prefill_split=3).info()
    assert sp["prefill_dynamic"] == (0 if sp["prefill_split_items"] > 0 else 1)
    small = workloads.make_batch([700, 300], [700, 900], num_q_heads=4, num_kv_heads=2,
                                 head_dim=256, page_size=128, windows=[0, 128], meta_only=True)
    sp = plan_of(small, prefill_split=3).info()
    assert sp["prefill_split_items"] > 0 and sp["prefill_dynamic"] == 0
    if name != "mixed":
        assert plan_of(b, prefill_pairs=2).info()["prefill_dynamic"] == 0


def test_dynamic_prefill_list_runs_in_l2_sized_groups():
    """When every prefill sequence sees its whole prefix (no window shorter
    than its KV), their K and V (kv_len x D x 2 x 2 bytes per (sequence, KV
    head)) exceed 1.5 x 40 MiB and every pair is read by at least four items
    on average, the dynamic list runs the pairs in ceil(total / 40 MiB)
    groups of equal bytes (pair order), longest first within each group;
    otherwise one group."""
    def want(b):
        ql = np.diff(b.cu_q_lens)
        pre = [s for s in range(b.num_seqs) if ql[s] > 1]
        per = [int(b.kv_lens[s]) * b.head_dim * 4 for s in pre for _ in range(b.num_kv_heads)]
        total = float(sum(per))
        items = len(prefill_items(b, plan_of(b).info()["q_block"])) * b.num_kv_heads
        windowed = any(b.window is not None and 0 < int(b.window[s]) < int(b.kv_lens[s])
                       for s in pre)
        if windowed or not (total > 1.5 * 40 * 2**20 and items >= 4 * len(per)):
            return 1
        return max(1, -(-int(total) // (40 * 2**20)))
    for name in ("causal_prefill", "swa_prefill", "mixed", "spec_decode"):
        b = workloads.WORKLOADS[name](meta_only=True)
        info = plan_of(b).info()
        assert info["prefill_groups"] == want(b), name
    # The causal 8k prefill: 16 heads x 8 MiB in four groups of four heads;
    # the sliding-window one, the mixed batch's four chunks (24 MiB) and
    # multi-token decode (one item per pair) in one.
    assert plan_of(workloads.WORKLOADS["causal_prefill"](meta_only=True)).info()["prefill_groups"] == 4
    assert plan_of(workloads.WORKLOADS["swa_prefill"](meta_only=True)).info()["prefill_groups"] == 1
    assert plan_of(workloads.WORKLOADS["mixed"](meta_only=True)).info()["prefill_groups"] == 1
    assert plan_of(workloads.WORKLOADS["spec_decode"](meta_only=True)).info()["prefill_groups"] == 1
    # Fixed lists have no groups; prefill_grouping = -1 keeps one.
    b = workloads.WORKLOADS["causal_prefill"](meta_only=True)
    assert plan_of(b, prefill_dynamic=-1).info()["prefill_groups"] == 0
    assert plan_of(b, prefill_grouping=-1).info()["prefill_groups"] == 1
    for bad in (-2, 1):
        with pytest.raises(RpaError) as e:
            plan_of(b, prefill_grouping=bad)
        assert e.value.status == binding.RPA_ERR_INVALID_ARG
