"""CPU oracle for ragged paged attention -- TEST INFRASTRUCTURE ONLY.

The plain definition of the attention step that the GPU library is checked
against (see ``rpa_oracle.cpp`` for the definition and its sources).  Only the
test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package.  It shares no code with ``ragged_paged_attention_rpa_gb300``
and imports nothing from it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rpa_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle_rpa.so")

_libs = {}

CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC"]


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle source into a shared library (default: next to it)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp.%d" % os.getpid()
    subprocess.run(["g++"] + CXXFLAGS + ["-o", tmp, src], check=True)
    os.replace(tmp, out)
    return out


def _load(lib_path=None):
    """Load the oracle library (``lib_path`` selects another build of it)."""
    key = lib_path or _LIB
    if key not in _libs:
        lib = ctypes.CDLL(build() if lib_path is None else lib_path)
        i32, i64, dbl, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        common = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, i32, vp, vp, vp, i32,
                  i32, i32, i32, i32, i32, dbl]
        lib.rpa_oracle_rows.argtypes = common + [vp, i64, vp, vp, ctypes.c_int]
        lib.rpa_oracle_rows.restype = ctypes.c_int
        lib.rpa_oracle_prow.argtypes = common + [i64, vp, vp, vp]
        lib.rpa_oracle_prow.restype = ctypes.c_int
        lib.rpa_oracle_round_bf16.argtypes = [vp, vp, i64]
        lib.rpa_oracle_round_bf16.restype = None
        _libs[key] = lib
    return _libs[key]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_inputs(q, k_pages, v_pages):
    """Accept uint16 arrays (bf16 bit patterns) or float32 arrays."""
    arrs = [np.ascontiguousarray(x) for x in (q, k_pages, v_pages)]
    dt = arrs[0].dtype
    if any(a.dtype != dt for a in arrs):
        raise TypeError("q, k_pages and v_pages must share a dtype")
    if dt == np.uint16:
        return 0, arrs
    if dt == np.float32:
        return 1, arrs
    raise TypeError("inputs must be uint16 (bf16 bits) or float32, got %s" % dt)


def _meta(page_table, cu_q_lens, kv_lens, window):
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    cu = np.ascontiguousarray(cu_q_lens, dtype=np.int32)
    kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
    win = None if window is None else np.ascontiguousarray(window, dtype=np.int32)
    return pt, cu, kl, win


def attention(q, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window,
              sm_scale, rows=None, precision=32, threads=0, with_bf16=False,
              lib_path=None):
    """Run the oracle.

    q: [total_q, Hq, D]; k_pages/v_pages: [num_pages, P, Hkv, D], as uint16 bf16
    bits or float32.  page_table: [num_seqs, max_pages_per_seq] int32.
    window: None, or int32 [num_seqs] (<= 0: full causal).
    rows: None for every row, else int64 indices r = token * Hq + head.
    Returns float64 [n_rows, D] (and the bf16-rounded uint16 copy if asked).
    """
    lib = _load(lib_path)
    in_dtype, (q, k, v) = _as_inputs(q, k_pages, v_pages)
    total_q, hq, d = q.shape
    num_pages, p, hkv, d2 = k.shape
    assert d2 == d and v.shape == k.shape
    pt, cu, kl, win = _meta(page_table, cu_q_lens, kv_lens, window)
    num_seqs = kl.shape[0]
    assert cu.shape[0] == num_seqs + 1 and pt.shape[0] == num_seqs
    if rows is None:
        n = total_q * hq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.shape[0]
    out = np.empty((n, d), dtype=np.float64)
    out16 = np.empty((n, d), dtype=np.uint16) if with_bf16 else None
    rc = lib.rpa_oracle_rows(precision, in_dtype, _ptr(q), _ptr(k), _ptr(v), _ptr(pt),
                             pt.shape[1], _ptr(cu), _ptr(kl), _ptr(win), num_seqs, hq,
                             hkv, d, p, num_pages, float(sm_scale), _ptr(rows_arr), n,
                             _ptr(out), _ptr(out16), threads)
    if rc != 0:
        raise ValueError("oracle rejected the problem (code %d)" % rc)
    return (out, out16) if with_bf16 else out


def softmax_row(q, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window,
                sm_scale, row, precision=32, lib_path=None):
    """Normalised softmax probabilities of one output row over its visible keys.

    Returns (p, lo, hi): p[j - lo] for visible keys lo..hi inclusive.
    """
    lib = _load(lib_path)
    in_dtype, (q, k, v) = _as_inputs(q, k_pages, v_pages)
    total_q, hq, d = q.shape
    num_pages, p_sz, hkv, _ = k.shape
    pt, cu, kl, win = _meta(page_table, cu_q_lens, kv_lens, window)
    num_seqs = kl.shape[0]
    buf = np.zeros(max(1, int(kl.max()) if num_seqs else 1), dtype=np.float64)
    lo = np.zeros(1, dtype=np.int64)
    hi = np.zeros(1, dtype=np.int64)
    rc = lib.rpa_oracle_prow(precision, in_dtype, _ptr(q), _ptr(k), _ptr(v), _ptr(pt),
                             pt.shape[1], _ptr(cu), _ptr(kl), _ptr(win), num_seqs, hq,
                             hkv, d, p_sz, num_pages, float(sm_scale), int(row),
                             _ptr(buf), _ptr(lo), _ptr(hi))
    if rc != 0:
        raise ValueError("oracle rejected the problem (code %d)" % rc)
    return buf[: int(hi[0] - lo[0]) + 1].copy(), int(lo[0]), int(hi[0])


def round_bf16(x):
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.rpa_oracle_round_bf16(_ptr(x), _ptr(out), x.size)
    return out


def write_kv(k_pages, v_pages, k_new, v_new, page_table, cu_q_lens, kv_lens):
    """The KV-cache write of a step's new tokens ("TPU Deep Dive" slides,
    chapter 8, "Continuous batching with static shapes": ragged paged
    attention writes the step's KV itself), as a plain loop: token
    t = cu_q_lens[s] + i of sequence s sits at position
    pos = kv_lens[s] - q_len + i, and its row for KV head g is copied to
    page page_table[s][pos // P], slot pos % P.  Returns new copies of the
    pools (any dtype; the copy is exact).  Parity pinned by
    tests/test_oracle_pins.py (pools rebuilt bitwise from their own rows)."""
    kp = np.array(k_pages, copy=True)
    vp = np.array(v_pages, copy=True)
    pt, cu, kl, _ = _meta(page_table, cu_q_lens, kv_lens, None)
    P = kp.shape[1]
    hkv = kp.shape[2]
    for s in range(kl.shape[0]):
        ql = int(cu[s + 1] - cu[s])
        for i in range(ql):
            t = int(cu[s]) + i
            pos = int(kl[s]) - ql + i
            page = int(pt[s, pos // P])
            for g in range(hkv):
                kp[page, pos % P, g, :] = k_new[t, g, :]
                vp[page, pos % P, g, :] = v_new[t, g, :]
    return kp, vp


def decode_e4m3(codes) -> np.ndarray:
    """OCP fp8 e4m3 codes -> float32, from the format's definition: sign bit,
    4-bit exponent with bias 7, 3-bit mantissa; exponent field 0 is
    subnormal (m/8 * 2^-6); S.1111.111 is NaN (no infinities)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    out = sign * mag
    out = np.where((e == 15) & (m == 7), np.nan, out)
    return out.astype(np.float32)


def dequantize_kv(codes, scale) -> np.ndarray:
    """fp8 pages [num_pages, P, Hkv, D] with a scale per KV head -> float32
    values (decoded code * scale of its head)."""
    vals = decode_e4m3(codes)
    return (vals * np.asarray(scale, dtype=np.float32)[None, None, :, None]).astype(np.float32)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rms_norm(x, weight, eps):
    """RMS normalisation over the last axis, in float64: x / sqrt(mean(x^2) +
    eps) * weight ("Chasing speed of light on TPU v6e", section "The Long
    Tail": the q/k/v RMS norms run right before attention).  weight None =
    no scaling."""
    x = np.asarray(x, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + float(eps))
    y = x * r
    if weight is not None:
        y = y * np.asarray(weight, dtype=np.float64)
    return y


def rope_angles(pos, head_dim, theta):
    """Rotation angles [len(pos), D/2] in float64: pos * theta^(-2i/D)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = np.power(float(theta), -2.0 * i / head_dim)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]


def rope(y, pos, theta):
    """Rotary position embedding of rows y [n, ..., D] at positions pos [n],
    float64, halves convention: dimension i < D/2 pairs with i + D/2 and the
    pair turns by the angle pos * theta^(-2i/D):
        out_i       = y_i cos a - y_{i+D/2} sin a
        out_{i+D/2} = y_{i+D/2} cos a + y_i sin a.
    theta <= 0: no rotation."""
    y = np.asarray(y, dtype=np.float64)
    if theta <= 0:
        return y.copy()
    D = y.shape[-1]
    a = rope_angles(pos, D, theta)
    shape = (a.shape[0],) + (1,) * (y.ndim - 2) + (D // 2,)
    c, s = np.cos(a).reshape(shape), np.sin(a).reshape(shape)
    lo, hi = y[..., : D // 2], y[..., D // 2:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def token_positions(cu_q_lens, kv_lens):
    """Position of every query token: kv_lens[s] - q_len_s + i."""
    cu = np.asarray(cu_q_lens, dtype=np.int64)
    kl = np.asarray(kv_lens, dtype=np.int64)
    pos = np.empty(int(cu[-1]), dtype=np.int64)
    for s in range(kl.shape[0]):
        ql = int(cu[s + 1] - cu[s])
        pos[cu[s]:cu[s + 1]] = kl[s] - ql + np.arange(ql)
    return pos


def qkv_prologue(q, k, v, q_weight, k_weight, v_weight, eps, theta, cu_q_lens, kv_lens):
    """The step before attention, as plain float64 math: q and k rows RMS-
    normalised (their weights; None = no norm) then rotated at their token's
    position; v rows RMS-normalised when v_weight is given, never rotated.
    q [T, Hq, D], k and v [T, Hkv, D] (any float dtype).  Returns float64
    (q_out, k_out, v_out); the caller rounds and writes k/v into pages."""
    pos = token_positions(cu_q_lens, kv_lens)

    def norm(x, w):
        return np.asarray(x, dtype=np.float64) if w is None else rms_norm(x, w, eps)

    q_out = rope(norm(q, q_weight), pos, theta)
    k_out = rope(norm(k, k_weight), pos, theta)
    v_out = norm(v, v_weight)
    return q_out, k_out, v_out
