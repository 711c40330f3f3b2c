"""GPU parity of the q/k/v prologue (rpa_qkv_prologue) and of the prologue
followed by attention (rpa_forward_qkv), through the C ABI, against the
float64 oracle.

Bounds: the kernel computes in fp32 and rounds its outputs once, so for bf16
every element is within 2^-8 of the oracle's value relative to itself plus
1e-5 of its row's largest magnitude (half a bf16 step is 2^-9; the rest
covers fp32 norm arithmetic and the rotation angle, which the kernel reduces
in extended precision); fp32 outputs are within 1e-5 of the row's largest
magnitude.  Pool slots other than the new tokens' stay bit for bit.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ragged_paged_attention_rpa_gb300 import binding, build, workloads

from .test_gpu_parity import assert_bf16_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def to_dev(a, dtype):
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(oracle.round_bf16(a.astype(np.float32)).view(np.int16)).view(
            torch.bfloat16).cuda()
    return torch.from_numpy(a.astype(np.float32)).cuda()


def from_dev(t):
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(
            np.float64)
    return t.cpu().numpy().astype(np.float64)


def assert_rows_close(got, want, dtype, what):
    scale = np.max(np.abs(want), axis=-1, keepdims=True)
    err = np.abs(got - want)
    if dtype == "bf16":
        bound = 2.0 ** -8 * np.abs(want) + 1e-5 * scale
    else:
        bound = 1e-5 * scale
    bad = err > bound
    assert not bad.any(), "%s: %d elements out of bound, worst excess %.3g" % (
        what, int(bad.sum()), float((err - bound).max()))


CASES = [
    # (q_lens, kv_lens, Hq, Hkv, D, P, dtype, weights (q, k, v), theta)
    ([1, 3, 1, 9], [40, 3, 700, 300], 8, 2, 128, 16, "bf16", (True, True, True), 10000.0),
    ([1] * 5, [129, 1, 4000, 77, 2048], 8, 1, 256, 128, "bf16", (True, True, False), 1e6),
    ([4, 2], [1000003, 999999], 4, 2, 64, 128, "bf16", (True, True, True), 10000.0),
    ([5, 1], [9, 2], 4, 4, 64, 32, "f32", (True, False, True), 500000.0),
    ([2, 7], [100000, 70], 16, 2, 256, 64, "f32", (False, True, False), 10000.0),
    ([3], [3], 2, 1, 128, 16, "bf16", (False, False, False), 0.0),
]


def make_case(case, seed):
    ql, kv, hq, hkv, d, p, dtype, (uq, uk, uv), theta = CASES[case]
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    kl = np.asarray(kv, dtype=np.int32)
    T = int(cu[-1])
    n = len(ql)
    # Each sequence owns distinct pages for its new tokens' slots; every other
    # page-table slot points at page 0.
    mpps = max(-(-L // p) for L in kv)
    slots = sorted({(s, pos // p) for s in range(n) for pos in range(kv[s] - ql[s], kv[s])})
    num_pages = len(slots) + 2
    ids = rng.permutation(np.arange(1, num_pages))[: len(slots)]
    pt = np.zeros((n, mpps), dtype=np.int32)
    for (s, sl), pg in zip(slots, ids):
        pt[s, sl] = pg
    q = rng.normal(size=(T, hq, d)) * 2.0
    k = rng.normal(size=(T, hkv, d)) * 0.5
    v = rng.normal(size=(T, hkv, d))
    w = [rng.uniform(0.5, 1.5, size=d) if use else None for use in (uq, uk, uv)]
    pool_k = rng.normal(size=(num_pages, p, hkv, d))
    pool_v = rng.normal(size=(num_pages, p, hkv, d))
    return dict(q=q, k=k, v=v, w=w, theta=theta, cu=cu, kl=kl, pt=pt, num_pages=num_pages,
                pool_k=pool_k, pool_v=pool_v, dtype=dtype, d=d, p=p)


def run_prologue(c, in_place=False, workspace=None):
    dt = c["dtype"]
    dq, dk, dv = (to_dev(c[x], dt) for x in ("q", "k", "v"))
    kp, vp = to_dev(c["pool_k"], dt), to_dev(c["pool_v"], dt)
    ws_ = [None if w is None else torch.from_numpy(w.astype(np.float32)).cuda() for w in c["w"]]
    norm = binding.qkv_norm(*ws_, eps=1e-6, rope_theta=c["theta"])
    qo = dq if in_place else torch.empty_like(dq)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda") if workspace is None else workspace
    binding.rpa_qkv_prologue(dq, dk, dv, norm, qo, kp, vp, torch.from_numpy(c["pt"]).cuda(),
                             torch.from_numpy(c["cu"]).cuda(), torch.from_numpy(c["kl"]).cuda(),
                             c["num_pages"], workspace=ws)
    torch.cuda.synchronize()
    return qo, kp, vp, ws


def inputs_as_stored(c):
    """The inputs as the device holds them (bf16-rounded for bf16 cases)."""
    if c["dtype"] == "bf16":
        return [oracle.bf16_bits_to_f32(oracle.round_bf16(c[x].astype(np.float32))).astype(
            np.float64) for x in ("q", "k", "v", "pool_k", "pool_v")]
    return [c[x].astype(np.float32).astype(np.float64) for x in ("q", "k", "v", "pool_k",
                                                                   "pool_v")]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prologue_matches_oracle(case):
    c = make_case(case, 900 + case)
    qo, kp, vp, ws = run_prologue(c)
    assert binding.rpa_get_device_error(ws) == 0
    q, k, v, pk, pv = inputs_as_stored(c)
    wq, wk, wv = (None if w is None else w.astype(np.float32).astype(np.float64) for w in c["w"])
    want_q, want_k, want_v = oracle.qkv_prologue(q, k, v, wq, wk, wv, 1e-6, c["theta"],
                                                 c["cu"], c["kl"])
    assert_rows_close(from_dev(qo), want_q, c["dtype"], "q_out case %d" % case)
    # The pools: new rows where the oracle's write puts them, the rest as before.
    exp_k, exp_v = oracle.write_kv(pk, pv, want_k, want_v, c["pt"], c["cu"], c["kl"])
    got_k, got_v = from_dev(kp), from_dev(vp)
    touched = np.zeros(pk.shape[:2], dtype=bool)
    pos = oracle.token_positions(c["cu"], c["kl"])
    for s in range(len(c["kl"])):
        for t in range(c["cu"][s], c["cu"][s + 1]):
            touched[c["pt"][s, pos[t] // c["p"]], pos[t] % c["p"]] = True
    assert np.array_equal(got_k[~touched], pk[~touched])
    assert np.array_equal(got_v[~touched], pv[~touched])
    assert_rows_close(got_k[touched], exp_k[touched], c["dtype"], "k rows case %d" % case)
    assert_rows_close(got_v[touched], exp_v[touched], c["dtype"], "v rows case %d" % case)


def test_prologue_in_place_q():
    c = make_case(0, 950)
    ref, _, _, _ = run_prologue(c)
    got, _, _, _ = run_prologue(c, in_place=True)   # q_out is q itself
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_prologue_reports_a_bad_page():
    c = make_case(0, 960)
    c["pt"] = c["pt"].copy()
    c["pt"][2, (c["kl"][2] - 1) // c["p"]] = c["num_pages"] + 3
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    _, kp, _, ws = run_prologue(c, workspace=ws)
    assert binding.rpa_get_device_error(ws) == binding.RPA_DEVERR_PAGE_ID


@pytest.mark.parametrize("name", ["decode", "spec_decode"])
def test_forward_qkv_matches_oracle(name):
    """Prologue then attention, against the oracle's prologue (rounded to bf16
    as stored), its KV write and its attention."""
    full = workloads.WORKLOADS[name](meta_only=True)
    keep = 16   # the first 16 sequences of the workload
    ql = np.diff(full.cu_q_lens)[:keep]
    b = workloads.make_batch(ql.tolist(), full.kv_lens[:keep].tolist(), num_q_heads=8,
                             num_kv_heads=1, head_dim=256, page_size=128, seed=970)
    rng = np.random.default_rng(971)
    T, D = b.total_q, b.head_dim
    qr = rng.normal(size=(T, 8, D))
    kr = rng.normal(size=(T, 1, D))
    vr = rng.normal(size=(T, 1, D))
    wq, wk = rng.uniform(0.5, 1.5, size=D), rng.uniform(0.5, 1.5, size=D)
    theta = 10000.0
    db = binding.Batch(b)
    plan = db.plan()
    ws = binding.alloc_workspace(plan)
    # The norm struct holds raw pointers: the weight tensors must outlive it.
    dwq = torch.from_numpy(wq.astype(np.float32)).cuda()
    dwk = torch.from_numpy(wk.astype(np.float32)).cuda()
    norm = binding.qkv_norm(dwq, dwk, None, eps=1e-6, rope_theta=theta)
    dq, dk, dv = (to_dev(x, "bf16") for x in (qr, kr, vr))
    q_buf = torch.empty_like(dq)
    binding.rpa_forward_qkv(dq, dk, dv, norm, q_buf, db.k_pages, db.v_pages, db.page_table,
                            db.cu_q_lens, db.kv_lens, db.window, b.sm_scale, db.out, plan, ws)
    assert binding.rpa_get_device_error(ws) == 0
    torch.cuda.synchronize()
    # Oracle: prologue on the stored (bf16) inputs, outputs rounded to bf16 as
    # the kernel stores them, written into the pools, then attention.
    q64, k64, v64 = (oracle.bf16_bits_to_f32(oracle.round_bf16(x.astype(np.float32))).astype(
        np.float64) for x in (qr, kr, vr))
    f32 = lambda x: x.astype(np.float32).astype(np.float64)   # noqa: E731
    oq, ok_, ov = oracle.qkv_prologue(q64, k64, v64, f32(wq), f32(wk), None, 1e-6, theta,
                                      b.cu_q_lens, b.kv_lens)
    rq, rk, rv = (oracle.round_bf16(x.astype(np.float32)) for x in (oq, ok_, ov))
    kp, vp = oracle.write_kv(b.k_pages, b.v_pages, rk, rv, b.page_table, b.cu_q_lens, b.kv_lens)
    want = oracle.attention(rq, kp, vp, b.page_table, b.cu_q_lens, b.kv_lens, b.window,
                            b.sm_scale, precision=32)
    got = db.out.float().cpu().numpy().reshape(-1, D).astype(np.float64)
    assert_bf16_close(got, want, "forward_qkv %s" % name)
