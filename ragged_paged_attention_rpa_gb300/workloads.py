"""Seeded synthetic inputs for ragged paged attention.

Shared by the tests and the benchmark.  This module only draws random numbers
and lays them out (lengths, page tables, bf16 tensors); it holds none of the
attention arithmetic and imports neither the oracle nor the CUDA library.

Shapes follow the workloads on the source pages:
  * "Chasing speed of light on TPU v6e", section "Attention": an 8192-token
    prefill whose sliding-window layers use a 1024-token window.
  * "Pallas kernel / vLLM on TPU ... 19,511 tokens per second", section
    "Strategy 3": eight query heads of dimension 256 share one KV head, and the
    cache is paged in 128-token blocks; batches of 128 to 512 decoding requests.
All values are N(0, 1) rounded to bf16 (or kept in float32 for the fp32 path).
No dataset is involved.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch


@dataclasses.dataclass
class Batch:
    name: str
    q: np.ndarray            # [total_q, Hq, D]   uint16 (bf16 bits) or float32
    k_pages: np.ndarray      # [num_pages, P, Hkv, D]
    v_pages: np.ndarray      # [num_pages, P, Hkv, D]
    page_table: np.ndarray   # [num_seqs, max_pages_per_seq] int32
    cu_q_lens: np.ndarray    # [num_seqs + 1] int32
    kv_lens: np.ndarray      # [num_seqs] int32
    window: Optional[np.ndarray]  # [num_seqs] int32 (<= 0: full causal) or None
    sm_scale: float
    seed: int
    # fp8 (e4m3) copies of the pools and their per-KV-head scales, when the
    # batch is meant for the fp8 decode path (see with_fp8_kv).
    k_fp8: Optional[np.ndarray] = None    # [num_pages, P, Hkv, D] uint8
    v_fp8: Optional[np.ndarray] = None
    k_scale: Optional[np.ndarray] = None  # [Hkv] float32
    v_scale: Optional[np.ndarray] = None

    @property
    def num_seqs(self) -> int:
        return int(self.kv_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k_pages.shape[2])

    @property
    def head_dim(self) -> int:
        return int(self.q.shape[2])

    @property
    def page_size(self) -> int:
        return int(self.k_pages.shape[1])

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def dtype(self) -> str:
        return "bf16" if self.q.dtype == np.uint16 else "f32"

    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_q_lens).astype(np.int32)


def _normal(rng: np.random.Generator, shape, dtype: str, meta_only: bool = False) -> np.ndarray:
    if meta_only:
        # Shape only (zero-stride, no memory): for scheduling tests that never
        # read the values.
        return np.broadcast_to(np.zeros((), np.uint16 if dtype == "bf16" else np.float32),
                               shape)
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if dtype == "f32":
        return x
    # bf16 via torch's round-to-nearest-even conversion, stored as raw bits.
    t = torch.from_numpy(x).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def make_batch(q_lens: Sequence[int], kv_lens: Sequence[int], *, num_q_heads: int,
               num_kv_heads: int, head_dim: int, page_size: int,
               windows: Optional[Sequence[int]] = None, seed: int = 0,
               pool_pages: Optional[int] = None, dtype: str = "bf16",
               sm_scale: Optional[float] = None, name: str = "batch",
               max_pages_per_seq: Optional[int] = None, meta_only: bool = False) -> Batch:
    """A ragged batch whose pages are drawn without replacement from a shuffled pool.

    Sequence s owns ceil(kv_lens[s] / page_size) pages; its page-table row is
    filled with distinct physical page ids taken from a random permutation of
    the pool.  Unused page-table slots hold -1 (never read).
    """
    q_lens = np.asarray(q_lens, dtype=np.int64)
    kv = np.asarray(kv_lens, dtype=np.int64)
    if q_lens.shape != kv.shape:
        raise ValueError("q_lens and kv_lens differ in length")
    if np.any(q_lens < 0) or np.any(kv < q_lens):
        raise ValueError("need 0 <= q_len <= kv_len for every sequence")
    ss = np.random.SeedSequence(seed)
    r_pool, r_q, r_k, r_v = [np.random.default_rng(c) for c in ss.spawn(4)]
    pages_per = (kv + page_size - 1) // page_size
    need = int(pages_per.sum())
    pool = need if pool_pages is None else int(pool_pages)
    if pool < need:
        raise ValueError("pool of %d pages cannot hold %d" % (pool, need))
    mpps = int(pages_per.max()) if len(kv) else 0
    if max_pages_per_seq is not None:
        mpps = max(mpps, int(max_pages_per_seq))
    mpps = max(mpps, 1)
    perm = r_pool.permutation(pool).astype(np.int32)
    table = np.full((len(kv), mpps), -1, dtype=np.int32)
    cur = 0
    for s, n in enumerate(pages_per):
        table[s, :n] = perm[cur:cur + n]
        cur += int(n)
    cu = np.zeros(len(kv) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    total_q = int(cu[-1])
    q = _normal(r_q, (total_q, num_q_heads, head_dim), dtype, meta_only)
    k = _normal(r_k, (pool, page_size, num_kv_heads, head_dim), dtype, meta_only)
    v = _normal(r_v, (pool, page_size, num_kv_heads, head_dim), dtype, meta_only)
    win = None if windows is None else np.asarray(windows, dtype=np.int32)
    scale = 1.0 / math.sqrt(head_dim) if sm_scale is None else float(sm_scale)
    return Batch(name, q, k, v, table, cu, kv.astype(np.int32), win, scale, seed)


# ---------------------------------------------------------------------------
# The five workloads.  Lengths are drawn from their own seeded stream, so the
# same seed always gives the same batch.


def tiny_prefill(seed: int = 0) -> Batch:
    """1 sequence, 256 queries over 256 keys, causal; 4 q / 1 kv heads, D 64;
    16-token pages, 16 pages in a randomly permuted pool of 32."""
    return make_batch([256], [256], num_q_heads=4, num_kv_heads=1, head_dim=64,
                      page_size=16, pool_pages=32, seed=seed,
                      sm_scale=1.0 / 8.0, name="tiny_prefill_256_h4kv1_d64_p16")


def decode_batch(seed: int = 1, num_seqs: int = 128, lo: int = 128, hi: int = 2048,
                 pool_pages: int = 4096, meta_only: bool = False) -> Batch:
    """128 decoding sequences (1 query each), KV length uniform in [128, 2048];
    8 q / 1 kv heads (MQA), D 256; 128-token pages from a shuffled pool of 4096."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 101]))
    kv = rng.integers(lo, hi + 1, size=num_seqs)
    return make_batch(np.ones(num_seqs, dtype=np.int64), kv, num_q_heads=8,
                      num_kv_heads=1, head_dim=256, page_size=128,
                      pool_pages=pool_pages, seed=seed, meta_only=meta_only,
                      name="decode_b%d_l%d-%d_h8kv1_d256_p128" % (num_seqs, lo, hi))


def spec_decode_batch(seed: int = 6, num_seqs: int = 128, spec: int = 8, lo: int = 128,
                      hi: int = 2048, pool_pages: int = 4096, meta_only: bool = False) -> Batch:
    """Multi-token (speculative) decode: the decode batch's shape with `spec`
    new tokens per sequence (the drafted tokens verified in one step), KV
    length uniform in [lo, hi] including them; 8 q / 1 kv heads, so one KV
    head serves spec x 8 = 64 query rows; D 256, 128-token pages."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 106]))
    kv = rng.integers(max(lo, spec), hi + 1, size=num_seqs)
    return make_batch(np.full(num_seqs, spec, dtype=np.int64), kv, num_q_heads=8,
                      num_kv_heads=1, head_dim=256, page_size=128, pool_pages=pool_pages,
                      seed=seed, meta_only=meta_only,
                      name="spec_decode_b%d_q%d_l%d-%d_h8kv1_d256_p128" % (num_seqs, spec, lo, hi))


def prefill_8k(seed: int = 2, window: int = 1024, tokens: int = 8192,
               num_q_heads: int = 32, num_kv_heads: int = 16, meta_only: bool = False) -> Batch:
    """One 8192-token sequence attending causally to itself; 32 q / 16 kv heads,
    D 256, 128-token pages randomly permuted.  window <= 0: global causal."""
    pages = (tokens + 127) // 128
    name = ("swa%d" % window if window > 0 else "causal") + \
        "_prefill_%d_h%dkv%d_d256_p128" % (tokens, num_q_heads, num_kv_heads)
    return make_batch([tokens], [tokens], num_q_heads=num_q_heads,
                      num_kv_heads=num_kv_heads, head_dim=256, page_size=128,
                      windows=[window], pool_pages=pages, seed=seed, name=name,
                      meta_only=meta_only)


def mixed_batch(seed: int = 4, num_decode: int = 512, num_prefill: int = 4,
                chunk: int = 2048, meta_only: bool = False) -> Batch:
    """512 decoding sequences (KV length uniform in [256, 4096]) followed by 4
    chunked-prefill sequences of 2048 new tokens appended to a prior length
    uniform in [0, 4096]; 8 q / 1 kv heads, D 256, 128-token pages, random
    permutation.  Sequences with an even index use window 1024, odd ones are
    full causal."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 105]))
    dec = rng.integers(256, 4096 + 1, size=num_decode)
    prior = rng.integers(0, 4096 + 1, size=num_prefill)
    kv = np.concatenate([dec, prior + chunk])
    ql = np.concatenate([np.ones(num_decode, dtype=np.int64),
                         np.full(num_prefill, chunk, dtype=np.int64)])
    n = num_decode + num_prefill
    win = np.where(np.arange(n) % 2 == 0, 1024, 0)
    need = int(((kv + 127) // 128).sum())
    return make_batch(ql, kv, num_q_heads=8, num_kv_heads=1, head_dim=256,
                      page_size=128, windows=win, pool_pages=need, seed=seed,
                      meta_only=meta_only, name="mixed_d%d_p%dx%d_h8kv1_d256_p128" % (num_decode, num_prefill,
                                                                  chunk))


WORKLOADS = {
    "tiny_prefill": tiny_prefill,
    "decode": decode_batch,
    "swa_prefill": lambda seed=2, **kw: prefill_8k(seed=seed, window=1024, **kw),
    "causal_prefill": lambda seed=3, **kw: prefill_8k(seed=seed, window=0, **kw),
    "mixed": mixed_batch,
    "spec_decode": spec_decode_batch,
}


def e4m3_encode(x) -> np.ndarray:
    """float -> OCP fp8 e4m3 codes (uint8): round to nearest even, saturating
    at +-448 (exponent bias 7, 3 mantissa bits, subnormals 2^-9 apart)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    e = np.clip(np.floor(np.log2(np.maximum(a, 2.0 ** -10))), -6, 8)
    q = np.minimum(np.round(a / 2.0 ** (e - 3)) * 2.0 ** (e - 3), 448.0)
    sub = q < 2.0 ** -6
    E = np.floor(np.log2(np.maximum(q, 2.0 ** -6)))
    m_norm = np.round(q / 2.0 ** E * 8.0 - 8.0)
    e_field = np.where(sub, 0, E + 7)
    m_field = np.where(sub, np.round(q / 2.0 ** -9), m_norm)
    code = (e_field.astype(np.uint8) << 3) | m_field.astype(np.uint8)
    return code | (np.signbit(x).astype(np.uint8) << 7)


def with_fp8_kv(b: Batch) -> Batch:
    """The batch with e4m3 copies of its K/V pools: per KV head, scale =
    max |value| / 448 over the pool, code = e4m3(value / scale)."""
    def quant(pool):
        if pool.dtype == np.uint16:                      # bf16 bits -> float32
            vals = (pool.astype(np.uint32) << 16).view(np.float32)
        else:
            vals = pool.astype(np.float32)
        hkv = pool.shape[2]
        scale = np.empty(hkv, dtype=np.float32)
        codes = np.empty(pool.shape, dtype=np.uint8)
        for g in range(hkv):
            m = float(np.abs(vals[:, :, g, :]).max())
            scale[g] = np.float32(m / 448.0 if m > 0 else 1.0)
            codes[:, :, g, :] = e4m3_encode(vals[:, :, g, :] / scale[g])
        return codes, scale
    kf, ks = quant(b.k_pages)
    vf, vs = quant(b.v_pages)
    return dataclasses.replace(b, name=b.name + "_fp8kv", k_fp8=kf, v_fp8=vf, k_scale=ks,
                               v_scale=vs)


WORKLOADS["decode_fp8"] = lambda seed=1, **kw: with_fp8_kv(decode_batch(seed=seed, **kw))
