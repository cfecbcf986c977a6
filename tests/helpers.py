"""Shared test helpers: turn a seeded Workload into oracle problems and compare."""
from __future__ import annotations

import numpy as np

import oracle
from gated_deltanet_linear_gdr_gb300 import workloads as W


def problem(w: W.Workload, state=None, **over) -> oracle.Problem:
    """An oracle.Problem over the workload's inputs; ``state`` defaults to the
    initial pool restricted to the live slots."""
    if state is None:
        state = w.state_pool(w.live_slots())
    kw = dict(nk=w.nk, nv=w.nv, K=w.K, V=w.V, decay_is_log=w.decay_is_log,
              use_l2norm=w.use_l2norm, scale=w.scale, eps=w.eps)
    kw.update(over)
    return oracle.Problem(w.qkv, w.decay, w.beta, state, w.slot_idx, w.offsets, **kw)


def state_f64(state: np.ndarray) -> np.ndarray:
    if state.dtype == np.uint16:
        return oracle.bf16_to_f64(state)
    return state.astype(np.float64)


def sub_workload(w: W.Workload, rows) -> W.Workload:
    """The same problem restricted to a subset of rows (rows are independent)."""
    rows = list(rows)
    L = w.row_lengths
    offs = [0]
    tok = []
    for b in rows:
        t0, t1 = int(w.offsets[b]), int(w.offsets[b + 1])
        tok.extend(range(t0, t1))
        offs.append(offs[-1] + (t1 - t0))
    tok = np.asarray(tok, dtype=np.int64)
    import dataclasses
    sub = dataclasses.replace(
        w, qkv=w.qkv[tok], decay=w.decay[tok], beta=w.beta[tok],
        slot_idx=w.slot_idx[rows].copy(), offsets=np.asarray(offs, dtype=np.int32),
        ring_slot_idx=None if w.ring_slot_idx is None else w.ring_slot_idx[rows].copy(),
        counts=None if w.counts is None else w.counts[rows].copy(),
        accepted=None if w.accepted is None else w.accepted[rows].copy())
    assert (sub.row_lengths == L[rows]).all()
    return sub


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of the bfloat16 grid at |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    a = np.maximum(a, 2.0 ** -126)
    e = np.floor(np.log2(a))
    return 2.0 ** (e - 7)
