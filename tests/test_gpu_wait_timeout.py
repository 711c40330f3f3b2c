"""Failure detection without a GPU fault: every wait inside librpa's kernels
is bounded (sm100_ptx.cuh, mbar_wait) and a wait that gives up raises the
CTA's abort flag and writes RPA_DEVERR_TIMEOUT into the workspace error word,
which the host reads with rpa_get_device_error; the kernel ends and the
context stays usable.  The test makes a wait run out on an mbarrier that
nothing arrives on (2 ms limit), and a second one end early when another warp
raises the abort flag."""

from __future__ import annotations

import ctypes
import os
import subprocess

import pytest
import torch

from ragged_paged_attention_rpa_gb300 import binding, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def helper(tmp_path_factory):
    build.build()
    lib = str(tmp_path_factory.mktemp("wait") / "libwaitcheck.so")
    src = os.path.join(os.path.dirname(__file__), "csrc", "wait_timeout_check.cu")
    subprocess.run([build.nvcc()] + build.ARCH + ["-O3", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I" + build.CSRC, "-I" + build.INCLUDE,
                    "-o", lib, src], check=True)
    L = ctypes.CDLL(lib)
    L.wait_timeout_check.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_ulonglong,
                                     ctypes.POINTER(ctypes.c_int)]
    return L


def run(L, limit_ns, peer_abort_ns):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    out = (ctypes.c_int * 3)()
    rc = L.wait_timeout_check(ctypes.c_void_p(ws.data_ptr()), limit_ns, peer_abort_ns, out)
    return rc, list(out), ws


def test_wait_gives_up_after_its_limit(helper):
    rc, (ok, aborted, us), ws = run(helper, 2_000_000, 0)
    assert rc == 0 and ok == 0 and aborted == 1
    assert 2000 <= us < 200000, us
    assert binding.rpa_get_device_error(ws) == binding.RPA_DEVERR_TIMEOUT
    assert binding.rpa_get_device_error(ws) == 0          # read and cleared
    # The context is still usable.
    assert torch.ones(4, device="cuda").sum().item() == 4.0


def test_wait_ends_when_another_warp_aborts(helper):
    rc, (ok, aborted, us), ws = run(helper, 2_000_000_000, 100_000)
    assert rc == 0 and ok == 0 and aborted == 1
    assert us < 100000, us                                # far below the 2 s limit
    assert binding.rpa_get_device_error(ws) == binding.RPA_DEVERR_TIMEOUT
