"""First calls from several host threads at once.

Each launcher looks up per-device facts (SM count, resident CTAs per SM, the
dynamic shared memory opt-in) on its first call and keeps them for later
calls.  This test starts a fresh process, so that every cache is cold, and
has several threads make their first calls of the three kernel families
(pipelined decode, short rows, general kernel) together, each on its own
stream; every result must equal the same call made alone afterwards, bit for
bit.  A thread that saw the cache marked ready before its values would launch
an empty grid and leave its output unwritten."""
from __future__ import annotations

import os
import subprocess
import sys
import threading

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _calls():
    """(name, workload, call) for one call of each kernel family; call(dev, ring)
    runs it and returns the output tensor."""
    from gated_deltanet_linear_gdr_gb300 import workloads as W

    dec = W.decode(batch=64, max_slots=80, n_pad=2)
    short = W.random_case(31, [5, 3, 0, 5, 4, 5], nk=4, nv=8, K=128, max_slots=8, state_dtype="bf16")
    long_ = W.random_case(32, [40, 3, 70, 0, 18], nk=2, nv=4, K=128, max_slots=6, state_dtype="bf16")
    return [
        ("decode", dec, lambda d, ring, rsi: d.fwd(max_row_len=1)),
        ("verify", short, lambda d, ring, rsi: d.verify(ring, rsi, max_row_len=5)),
        ("prefill", long_, lambda d, ring, rsi: d.fwd(max_row_len=0)),
    ]


def _child():
    import torch

    import gated_deltanet_linear_gdr_gb300 as gdr
    from tests.gpu_helpers import DEV, Dev, pool_to_host, ring_for

    calls = _calls()
    per_kind = 3
    jobs = []
    for name, w, call in calls:
        pool = w.state_pool()
        for _ in range(per_kind + 1):  # the last copy runs alone afterwards
            jobs.append((name, Dev(w, pool), ring_for(w, 8, w.batch),
                         torch.arange(w.batch, dtype=torch.int32, device=DEV), call))
    torch.cuda.synchronize()
    threaded = [j for i, j in enumerate(jobs) if i % (per_kind + 1) != per_kind]
    alone = [j for i, j in enumerate(jobs) if i % (per_kind + 1) == per_kind]
    results = {}
    gate = threading.Barrier(len(threaded))
    errors = []

    def run(i, job):
        name, d, ring, rsi, call = job
        try:
            s = torch.cuda.Stream(DEV)
            gate.wait()
            with torch.cuda.stream(s):
                out = call(d, ring, rsi)
            s.synchronize()
            results[i] = (name, out.cpu().numpy(), pool_to_host(d.state))
        except Exception as e:  # reported by the parent
            errors.append(f"{name}: {e!r}")

    threads = [threading.Thread(target=run, args=(i, j)) for i, j in enumerate(threaded)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    ref = {}
    for name, d, ring, rsi, call in alone:
        out = call(d, ring, rsi)
        torch.cuda.synchronize()
        ref[name] = (out.cpu().numpy(), pool_to_host(d.state))
    assert len(results) == len(threaded)
    for name, out, state in results.values():
        r_out, r_state = ref[name]
        assert not np.isnan(r_out).any(), name
        assert (out.view(np.uint32) == r_out.view(np.uint32)).all(), name
        assert (state == r_state).all(), name
    st = gdr.gdr_get_status(clear=True)
    assert st == 0, gdr.status_names(st)
    print("threads ok", len(threaded))


def test_first_calls_from_several_threads_at_once():
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", "import tests.test_gpu_threads as t; t._child()"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok 9" in r.stdout
