"""rpa_forward from several host threads at once: each call stages its
launch parameters in per-thread buffers, so concurrent calls on their own
streams (ctypes releases the GIL during the call) give exactly the results
they give one at a time."""

from __future__ import annotations

import threading

import numpy as np
import pytest
import torch

from ragged_paged_attention_rpa_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def batches():
    rng = np.random.default_rng(77)
    out = []
    for i in range(4):
        n = 40 + 10 * i
        kv = rng.integers(20, 3000, size=n).tolist()
        ql = [1] * (n - 2) + [50 + i, 200]
        kv[-2:] = [max(kv[-2], 60), max(kv[-1], 300)]
        out.append(workloads.make_batch(ql, kv, num_q_heads=8, num_kv_heads=1, head_dim=256,
                                        page_size=128, windows=[0 if j % 2 else 512 for j in range(n)],
                                        seed=1100 + i))
    return out


def test_concurrent_forward_calls_match_serial_ones():
    bs = batches()
    dbs = [binding.Batch(b) for b in bs]
    plans = [db.plan() for db in dbs]
    wss = [binding.alloc_workspace(p) for p in plans]
    serial = []
    for db, p, ws in zip(dbs, plans, wss):
        serial.append(db.forward(p, ws).clone())
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in bs]
    for db in dbs:
        db.out.zero_()
    torch.cuda.synchronize()
    errors = []

    def worker(i):
        try:
            torch.cuda.set_device(0)        # the thread's current device, as a caller sets it
            with torch.cuda.stream(streams[i]):
                call = dbs[i].call(plans[i], wss[i], stream=streams[i])
                for _ in range(20):
                    call()
        except Exception as e:  # noqa: BLE001
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(bs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i, (db, ws) in enumerate(zip(dbs, wss)):
        assert binding.rpa_get_device_error(ws) == 0
        assert torch.equal(db.out.view(torch.int16), serial[i].view(torch.int16)), i
