"""Contracts the pages state exactly, checked GPU against GPU, bit for bit:
verify writes the forward pass's output and leaves the pool alone; verify +
fold over a prefix equals the forward pass over it (float32 ring); long rows
commit like the forward pass; snapshots and rollback equal the forward pass
over the draft prefix; and the library's own guarantees (kernel choice,
batch composition, strides and repeated runs do not change any bit)."""
from __future__ import annotations

import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import gated_deltanet_linear_gdr_gb300 as gdr
import gated_deltanet_linear_gdr_gb300._binding as B
from gated_deltanet_linear_gdr_gb300 import workloads as W
from tests.gpu_helpers import DEV, Dev, pool_to_dev, pool_to_host, ring_for
from tests.helpers import sub_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    gdr.gdr_get_status(clear=True)
    yield


def _prefix(w, b, n):
    """Row b of w cut to its first n tokens, as a one-row workload."""
    sub = sub_workload(w, [b])
    return dataclasses.replace(sub, offsets=np.array([0, n], np.int32), qkv=sub.qkv[:n],
                               decay=sub.decay[:n], beta=sub.beta[:n])


def _run_fwd(w, pool, max_row_len=0):
    d = Dev(w, pool)
    out = d.fwd(max_row_len=max_row_len)
    torch.cuda.synchronize()
    return out.cpu().numpy(), pool_to_host(d.state)


@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
def test_verify_output_equals_forward_and_pool_untouched(state_dtype):
    w = W.verify_fold(batch=24, max_slots=48, ring_rows=48, state_dtype=state_dtype)
    pool = w.state_pool()
    out_f, pool_f = _run_fwd(w, pool)
    d = Dev(w, pool)
    ring = ring_for(w, w.ring_len, w.ring_rows)
    out_v = d.verify(ring, torch.from_numpy(w.ring_slot_idx).to(DEV)).cpu().numpy()
    assert (out_v.view(np.uint32) == out_f.view(np.uint32)).all()
    host = pool_to_host(d.state)
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        if w.row_lengths[b] > w.ring_len:
            assert (host[s] == pool_f[s]).all(), "long row must commit exactly like fwd"
            assert torch.isnan(ring[int(w.ring_slot_idx[b])]).all(), "long row must not record"
        else:
            assert (host[s] == pool[s]).all(), "verify must leave the pool alone"


def test_prepared_calls_replay_from_a_cuda_graph():
    """The entry points never synchronise or read device memory on the host, so
    a decode step and a verify + fold window captured into a CUDA graph replay
    with the same bits as direct calls."""
    w = W.decode(batch=64, max_slots=128)
    pool = w.state_pool()
    direct = Dev(w, pool)
    out_direct = direct.fwd(max_row_len=1).clone()
    captured = Dev(w, pool)
    out = torch.empty_like(out_direct)
    call = gdr.prepare_fwd(captured.qkv, captured.decay, captured.beta, captured.state, captured.slot,
                           captured.off, out, max_row_len=1)
    call()  # warm-up outside the graph (loads the library, sets kernel attributes)
    torch.cuda.synchronize()
    captured.state.copy_(pool_to_dev(pool))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    g.replay()
    torch.cuda.synchronize()
    assert (out.view(torch.int32) == out_direct.view(torch.int32)).all()
    assert (pool_to_host(captured.state) == pool_to_host(direct.state)).all()

    wv = W.verify_fold(batch=16, max_slots=32, ring_rows=32)
    pv = wv.state_pool()
    res = []
    for use_graph in (False, True):
        d = Dev(wv, pv)
        ring = ring_for(wv, wv.ring_len, wv.ring_rows)
        rsi = torch.from_numpy(wv.ring_slot_idx).to(DEV)
        o = torch.empty((wv.total_tokens, wv.nv * wv.V), device=DEV)
        v = gdr.prepare_verify_ring(d.qkv, d.decay, d.beta, d.state, d.slot, d.off, ring, rsi, o,
                                    max_row_len=12)
        f = gdr.prepare_fold(d.state, d.slot, ring, rsi, torch.from_numpy(wv.counts).to(DEV))
        if use_graph:
            v()
            f()
            torch.cuda.synchronize()
            d.state.copy_(pool_to_dev(pv))
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2):
                v()
                f()
            g2.replay()
        else:
            v()
            f()
        torch.cuda.synchronize()
        res.append((o.cpu().numpy(), pool_to_host(d.state)))
    assert (res[0][0].view(np.uint32) == res[1][0].view(np.uint32)).all()
    assert (res[0][1] == res[1][1]).all()
    assert gdr.gdr_get_status(clear=True) == 0


@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
def test_value_head_twice_key_head_equals_two_halves(state_dtype):
    """The value columns never mix: a V = 2K pass gives, bit for bit, the two
    V = K passes on the halves of the value columns."""
    K = 128
    w = W.random_case(820, [19, 2, 1], nk=2, nv=4, K=K, V=2 * K, max_slots=6, state_dtype=state_dtype)
    pool = w.state_pool()
    out, after = _run_fwd(w, pool)
    nv, qk = w.nv, 2 * w.nk * K
    for half in range(2):
        cols = slice(half * K, (half + 1) * K)
        v = w.qkv[:, qk:].reshape(-1, nv, 2 * K)[:, :, cols].reshape(-1, nv * K)
        wh = dataclasses.replace(w, V=K, qkv=np.ascontiguousarray(np.concatenate([w.qkv[:, :qk], v], axis=1)))
        out_h, after_h = _run_fwd(wh, np.ascontiguousarray(pool[..., cols]))
        assert (out.reshape(-1, nv, 2 * K)[:, :, cols].view(np.uint32) ==
                out_h.reshape(-1, nv, K).view(np.uint32)).all()
        assert (after[..., cols] == after_h).all()


@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
def test_key_head_twice_value_head_equals_half_of_a_square_pass(state_dtype):
    """A V = K/2 pass is, bit for bit, the first half of the value columns of a
    V = K pass whose other columns hold anything: columns never mix."""
    K = 128
    for hint, lengths in ((0, [19, 2, 1, 40]), (16, [16, 2, 1, 9]), (8, [8, 2, 0, 5])):
        w = W.random_case(821 + hint, lengths, nk=2, nv=4, K=K, max_slots=6, state_dtype=state_dtype)
        pool = w.state_pool()
        out, after = _run_fwd(w, pool, max_row_len=hint)
        nv, qk, H = w.nv, 2 * w.nk * K, K // 2
        v = w.qkv[:, qk:].reshape(-1, nv, K)[:, :, :H].reshape(-1, nv * H)
        wh = dataclasses.replace(w, V=H, qkv=np.ascontiguousarray(np.concatenate([w.qkv[:, :qk], v], axis=1)))
        out_h, after_h = _run_fwd(wh, np.ascontiguousarray(pool[..., :H]), max_row_len=hint)
        assert (out.reshape(-1, nv, K)[:, :, :H].view(np.uint32) == out_h.reshape(-1, nv, H).view(np.uint32)).all()
        assert (after[..., :H] == after_h).all()


@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
def test_dense_state_equals_pool_at_the_rows_slots(state_dtype):
    """The dense mode is the slot-indexed pass with the rows' states gathered:
    same output bits, final[b] = the pool slot of row b after the pass; also
    when the start and end buffers are the same tensor."""
    w = W.random_case(710, [17, 3, 1, 33], nk=2, nv=4, K=128, max_slots=9, state_dtype=state_dtype)
    pool = w.state_pool()
    out_pool, pool_after = _run_fwd(w, pool)
    init = pool_to_dev(pool[w.slot_idx])
    d = Dev(w, pool)
    out, final = gdr.gdr_fwd_dense(d.qkv, d.decay, d.beta, d.off, init)
    torch.cuda.synchronize()
    assert (out.cpu().numpy().view(np.uint32) == out_pool.view(np.uint32)).all()
    assert (pool_to_host(final) == pool_after[w.slot_idx]).all()
    # in place: one buffer as start and end state, through the C entry point
    a = gdr._binding.make_args(d.qkv, d.decay, d.beta, init, torch.zeros(w.batch, dtype=torch.int32,
                               device=DEV), d.off, out, nk=w.nk)
    gdr._binding._check(gdr.load_library().gdr_fwd_dense(
        ctypes.byref(a), init.data_ptr(), init.data_ptr(), torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert (pool_to_host(init) == pool_after[w.slot_idx]).all()
    assert (out.cpu().numpy().view(np.uint32) == out_pool.view(np.uint32)).all()


@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
def test_beta_per_value_constant_along_v_equals_headwise(state_dtype):
    """Per-element beta that is constant along V gives the head-wise result bit
    for bit (same operation on every column)."""
    w = W.random_case(620, [17, 3, 1], nk=2, nv=4, K=128, max_slots=6, state_dtype=state_dtype)
    pool = w.state_pool()
    out_h, pool_h = _run_fwd(w, pool)
    wp = dataclasses.replace(w, beta=np.repeat(w.beta[:, :, None], w.V, axis=2).copy())
    out_p, pool_p = _run_fwd(wp, pool)
    assert (out_h.view(np.uint32) == out_p.view(np.uint32)).all()
    assert (pool_h == pool_p).all()


@pytest.mark.parametrize("hint", [0, 12])  # general kernel / short-row kernel
def test_bf16_ring_verify_matches_f32_ring_verify(hint):
    """The ring dtype changes only the records: same output, same pool, and the
    bfloat16 records are the float32 records rounded to nearest-even."""
    w = W.verify_fold(batch=24, max_slots=48, ring_rows=48, nk=4, nv=8)
    pool = w.state_pool()
    rsi = torch.from_numpy(w.ring_slot_idx).to(DEV)
    res = []
    for dt in (torch.float32, torch.bfloat16):
        d = Dev(w, pool)
        ring = ring_for(w, w.ring_len, w.ring_rows, dt)
        out = d.verify(ring, rsi, max_row_len=hint)
        torch.cuda.synchronize()
        res.append((out.cpu().numpy(), pool_to_host(d.state), ring))
    assert (res[0][0].view(np.uint32) == res[1][0].view(np.uint32)).all()
    assert (res[0][1] == res[1][1]).all()
    r32, r16 = res[0][2], res[1][2]
    written = ~torch.isnan(r32)
    assert (written == ~torch.isnan(r16)).all()
    # compare written fields only (torch's NaN conversion picks its own bits)
    assert (r32.to(torch.bfloat16).view(torch.int16)[written] == r16.view(torch.int16)[written]).all()


@pytest.mark.parametrize("K", [32, 64, 128])
@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
def test_verify_plus_fold_equals_forward_over_prefix(state_dtype, K):
    kw = {} if K == 128 else dict(nk=2, nv=4, K=K)
    w = W.verify_fold(batch=24, max_slots=48, ring_rows=48, state_dtype=state_dtype, **kw)
    counts = np.array([b % 6 for b in range(w.batch)], np.int32)
    counts[-1] = w.row_lengths[-1]
    w = dataclasses.replace(w, counts=counts)
    pool = w.state_pool()
    d = Dev(w, pool)
    ring = ring_for(w, w.ring_len, w.ring_rows)
    rsi = torch.from_numpy(w.ring_slot_idx).to(DEV)
    d.verify(ring, rsi)
    gdr.gdr_fold(d.state, d.slot, ring, rsi, torch.from_numpy(counts).to(DEV))
    torch.cuda.synchronize()
    host = pool_to_host(d.state)
    _, pool_full = _run_fwd(w, pool)
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        c = int(counts[b])
        if w.row_lengths[b] > w.ring_len:
            assert (host[s] == pool_full[s]).all()
            continue
        if c == 0:
            assert (host[s] == pool[s]).all()
            continue
        _, pool_pref = _run_fwd(_prefix(w, b, c), pool)
        assert (host[s] == pool_pref[s]).all(), f"row {b} count {c}"


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_snapshots_and_rollback_equal_forward_over_prefix(state_dtype):
    w = W.gdp_snapshots(batch=6, max_slots=12, state_dtype=state_dtype)
    pool = w.state_pool()
    d = Dev(w, pool)
    tdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
    inter = torch.zeros((w.max_slots, w.n_inter, w.nv, w.K, w.V), dtype=tdt, device=DEV)
    out_s = d.snapshots(inter, w.steps_per_token).cpu().numpy()
    host_inter = pool_to_host(inter)
    final = pool_to_host(d.state)
    out_f, pool_f = _run_fwd(w, pool)
    assert (out_s.view(np.uint32) == out_f.view(np.uint32)).all()
    assert (final == pool_f).all()
    M = w.steps_per_token
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        for i in range(w.n_inter):
            _, pp = _run_fwd(_prefix(w, b, (i + 1) * M), pool)
            assert (host_inter[s, i] == pp[s]).all(), (b, i)
        assert (host_inter[s, w.n_inter - 1] == final[s]).all()
    acc = torch.from_numpy(w.accepted).to(DEV)
    gdr.gdr_rollback(d.state, d.slot, inter, acc)
    host = pool_to_host(d.state)
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        _, pp = _run_fwd(_prefix(w, b, (int(w.accepted[b]) + 1) * M), pool)
        assert (host[s] == pp[s]).all()


def test_chaining_float32_pool():
    """float32 pool: one call over L tokens == two calls over L1 and L - L1."""
    w = W.random_case(600, [23, 40], nk=2, nv=4, K=128, max_slots=4, state_dtype="f32")
    pool = w.state_pool()
    out, full = _run_fwd(w, pool)
    st = pool.copy()
    cuts = [10, 17]
    parts = []
    for first in (True, False):
        rows = []
        for b in range(w.batch):
            t0, t1 = int(w.offsets[b]), int(w.offsets[b + 1])
            c = t0 + cuts[b]
            rows.append((t0, c) if first else (c, t1))
        toks = np.concatenate([np.arange(a, z) for a, z in rows])
        offs = np.concatenate([[0], np.cumsum([z - a for a, z in rows])]).astype(np.int32)
        part = dataclasses.replace(w, qkv=w.qkv[toks], decay=w.decay[toks], beta=w.beta[toks],
                                   offsets=offs)
        o, st = _run_fwd(part, st)
        parts.append((o, rows))
    assert (st == full).all()


def test_decode_kernel_equals_general_kernel():
    w = W.decode(batch=48, max_slots=96)
    pool = w.state_pool()
    o1, s1 = _run_fwd(w, pool, max_row_len=1)
    o2, s2 = _run_fwd(w, pool, max_row_len=0)
    assert (o1.view(np.uint32) == o2.view(np.uint32)).all()
    assert (s1 == s2).all()


def test_batch_composition_does_not_change_bits():
    w = W.random_case(601, [5, 31, 1, 12], nk=2, nv=4, K=64, max_slots=6, state_dtype="bf16")
    pool = w.state_pool()
    out, st = _run_fwd(w, pool)
    for b in range(w.batch):
        o, s = _run_fwd(sub_workload(w, [b]), pool)
        t0, t1 = int(w.offsets[b]), int(w.offsets[b + 1])
        assert (o.view(np.uint32) == out[t0:t1].view(np.uint32)).all()
        assert (s[w.slot_idx[b]] == st[w.slot_idx[b]]).all()


def test_repeated_runs_are_identical():
    w = W.random_case(602, [17, 9], nk=2, nv=4, K=128, max_slots=4, state_dtype="bf16")
    pool = w.state_pool()
    a = _run_fwd(w, pool)
    b = _run_fwd(w, pool)
    assert (a[0].view(np.uint32) == b[0].view(np.uint32)).all() and (a[1] == b[1]).all()


def test_strided_views_equal_contiguous():
    """qkv, decay/beta and out as views with padded strides; a pool with padded
    rows -- same bits as the dense call."""
    w = W.random_case(603, [6, 19], nk=2, nv=4, K=64, max_slots=4, state_dtype="bf16")
    pool = w.state_pool()
    out_ref, st_ref = _run_fwd(w, pool)
    T, C = w.qkv.shape
    big = torch.zeros((T, C + 36), device=DEV)
    big[:, 4:4 + C] = torch.from_numpy(w.qkv).to(DEV)
    qkv = big[:, 4:4 + C]
    db = torch.zeros((T, 2 * w.nv + 8), device=DEV)
    db[:, :w.nv] = torch.from_numpy(w.decay).to(DEV)
    decay = db[:, :w.nv]
    bb = torch.zeros((T, 2 * w.nv + 8), device=DEV)
    bb[:, 3:3 + w.nv] = torch.from_numpy(w.beta).to(DEV)
    beta = bb[:, 3:3 + w.nv]
    ob = torch.zeros((T, w.nv * w.V * 2), device=DEV)
    out = ob[:, ::2]  # value-dim stride 2 (scalar stores)
    sbig = torch.zeros((w.max_slots, w.nv, w.K, w.V + 8), dtype=torch.bfloat16, device=DEV)
    sbig[..., :w.V] = pool_to_dev(pool)
    state = sbig[..., :w.V]
    gdr.gdr_fwd(qkv, decay, beta, state, torch.from_numpy(w.slot_idx).to(DEV),
                torch.from_numpy(w.offsets).to(DEV), out=out)
    torch.cuda.synchronize()
    assert (out.cpu().numpy().view(np.uint32) == out_ref.view(np.uint32)).all()
    assert (pool_to_host(state.contiguous()) == st_ref).all()


def test_beta0_decay1_leaves_bf16_state_bitwise():
    w = W.random_case(604, [7, 1], nk=1, nv=2, K=128, max_slots=3, state_dtype="bf16")
    w = dataclasses.replace(w, decay=np.ones_like(w.decay), beta=np.zeros_like(w.beta))
    pool = w.state_pool()
    _, st = _run_fwd(w, pool)
    assert (st == pool).all()
    _, st = _run_fwd(dataclasses.replace(w, offsets=np.array([0, 1, 2], np.int32),
                                         qkv=w.qkv[:2], decay=w.decay[:2], beta=w.beta[:2]),
                     pool, max_row_len=1)
    assert (st == pool).all()


def test_padding_rows_write_nothing_but_zero_output():
    w = W.random_case(605, [4, 3, 2], nk=2, nv=4, K=32, max_slots=5, state_dtype="f32")
    w = dataclasses.replace(w, slot_idx=np.array([1, -1, 3], np.int32))
    pool = w.state_pool()
    d = Dev(w, pool)
    out = torch.full((w.total_tokens, w.nv * w.V), float("nan"), device=DEV)
    d.fwd(out=out)
    ring = ring_for(w, 8, 5)
    d2 = Dev(w, pool)
    out2 = d2.verify(ring, torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV))
    inter = torch.full((5, 2, w.nv, w.K, w.V), float("nan"), device=DEV)
    d3 = Dev(w, pool)
    out3 = d3.snapshots(inter, 1)
    torch.cuda.synchronize()
    for o in (out, out2, out3):
        assert (o[4:7] == 0).all()
    for dd in (d, d2, d3):
        assert (pool_to_host(dd.state)[[0, 2, 4]] == pool[[0, 2, 4]]).all()
    assert torch.isnan(ring[1]).all()
    assert torch.isnan(inter[[0, 2, 4]]).all()


def test_device_status_flags_bad_inputs():
    w = W.random_case(606, [2, 1, 3], nk=1, nv=2, K=16, max_slots=4, state_dtype="f32")
    pool = w.state_pool()
    bad = dataclasses.replace(w, slot_idx=np.array([0, 9, 2], np.int32))
    d = Dev(bad, pool)
    out = torch.full((w.total_tokens, w.nv * w.V), float("nan"), device=DEV)
    d.fwd(out=out)
    st = gdr.gdr_get_status(clear=True)
    assert st & 0x1, gdr.status_names(st)
    assert (out[2:3] == 0).all()                     # the bad row's output is zeroed
    assert (pool_to_host(d.state)[[1, 3]] == pool[[1, 3]]).all()
    d = Dev(w, pool)
    out = torch.full((w.total_tokens, w.nv * w.V), float("nan"), device=DEV)
    d.fwd(max_row_len=2, out=out)                     # a row of 3 tokens breaks the bound
    st = gdr.gdr_get_status(clear=True)
    assert st & 0x10, gdr.status_names(st)
    assert (out[3:6] == 0).all()                     # ... and its output is zeroed
    assert gdr.gdr_get_status(clear=True) == 0


@pytest.mark.parametrize("K,state_dtype", [(16, "f32"), (128, "bf16"), (128, "f32")])
def test_row_longer_than_bound_zeroes_its_output(K, state_dtype):
    """A row longer than the caller's max_row_len is skipped by the forward,
    verify and snapshot passes (short-row kernel at K = 128, general kernel at
    K = 16): its output rows are zeroed, its slot, ring row and snapshots are
    left alone, ROW_TOO_LONG is flagged, and the other rows keep the bits of
    an unbounded call."""
    w = W.random_case(607, [2, 1, 3], nk=1, nv=2, K=K, max_slots=4, state_dtype=state_dtype)
    pool = w.state_pool()
    o_ref, s_ref = _run_fwd(w, pool)
    s2 = int(w.slot_idx[2])

    def nan_out():
        return torch.full((w.total_tokens, w.nv * w.V), float("nan"), device=DEV)

    def check(out):
        st = gdr.gdr_get_status(clear=True)
        assert st == 0x10, gdr.status_names(st)
        o = out.cpu().numpy()
        assert (o[3:6] == 0).all()
        assert (o[:3].view(np.uint32) == o_ref[:3].view(np.uint32)).all()

    d = Dev(w, pool)
    out = nan_out()
    d.fwd(max_row_len=2, out=out)
    check(out)
    host = pool_to_host(d.state)
    assert (host[s2] == pool[s2]).all()
    for b in (0, 1):
        s = int(w.slot_idx[b])
        assert (host[s] == s_ref[s]).all()

    d = Dev(w, pool)
    out = nan_out()
    ring = ring_for(w, 4, 3)
    d.verify(ring, torch.arange(3, dtype=torch.int32, device=DEV), max_row_len=2, out=out)
    check(out)
    assert torch.isnan(ring[2]).all()
    assert (pool_to_host(d.state) == pool).all()

    d = Dev(w, pool)
    out = nan_out()
    tdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
    inter = torch.full((w.max_slots, 3, w.nv, w.K, w.V), float("nan"), dtype=tdt, device=DEV)
    d.snapshots(inter, 1, max_row_len=2, out=out)
    check(out)
    assert torch.isnan(inter[s2].float()).all()
    assert (pool_to_host(d.state)[s2] == pool[s2]).all()


@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
def test_pipelined_decode_equals_simple_decode(state_dtype):
    """Unit-stride, aligned q/k/v rows take the pipelined decode kernel; a
    misaligned view of the same values takes the simple one: same bits."""
    w = W.decode(batch=96, max_slots=192, state_dtype=state_dtype)
    pool = w.state_pool()
    o1, s1 = _run_fwd(w, pool, max_row_len=1)
    d = Dev(w, pool)
    T, C = w.qkv.shape
    buf = torch.zeros(T * C + 1, device=DEV)
    buf[1:] = torch.from_numpy(w.qkv).to(DEV).reshape(-1)
    qkv = buf[1:].view(T, C)  # base 4 bytes past a 16-byte boundary
    out = gdr.gdr_fwd(qkv, d.decay, d.beta, d.state, d.slot, d.off, max_row_len=1)
    torch.cuda.synchronize()
    assert (out.cpu().numpy().view(np.uint32) == o1.view(np.uint32)).all()
    assert (pool_to_host(d.state) == s1).all()


def test_decode_kernel_device_checks():
    w = W.decode(batch=40, max_slots=64)
    pool = w.state_pool()
    slots = w.slot_idx.copy()
    live = np.flatnonzero(slots >= 0)
    slots[live[0]] = 1000  # beyond max_slots
    bad = dataclasses.replace(w, slot_idx=slots)
    d = Dev(bad, pool)
    out = torch.full((w.total_tokens, w.nv * w.V), float("nan"), device=DEV)
    d.fwd(max_row_len=1, out=out)
    st = gdr.gdr_get_status(clear=True)
    assert st & 0x1, gdr.status_names(st)
    b = int(live[0])
    assert (out[b] == 0).all()
    assert not torch.isnan(out).any()
    # a row of two tokens under max_row_len=1 is skipped and flagged
    offs = np.concatenate([[0], np.arange(2, w.batch + 1)]).astype(np.int32)  # row 0 has 2 tokens
    two = dataclasses.replace(w, offsets=offs, slot_idx=w.slot_idx[:-1].copy())
    d = Dev(two, pool)
    out = torch.full((w.total_tokens, w.nv * w.V), float("nan"), device=DEV)
    d.fwd(max_row_len=1, out=out)
    st = gdr.gdr_get_status(clear=True)
    assert st & 0x10, gdr.status_names(st)
    assert (out[0:2] == 0).all()  # the skipped row's two tokens
    assert not torch.isnan(out).any()
    s0 = int(two.slot_idx[0])
    if s0 >= 0:
        assert (pool_to_host(d.state)[s0] == pool[s0]).all()


@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
def test_short_row_kernel_equals_general_kernel(state_dtype):
    """The same rows through the short-row kernel (max_row_len hint) and the
    general kernel: forward, verify (records and pool) and snapshots agree bit
    for bit, including rows longer than one staged chunk."""
    lengths = [5, 1, 8, 0, 12, 3, 20, 7]
    w = W.random_case(700, lengths, nk=4, nv=8, K=128, max_slots=12, state_dtype=state_dtype,
                      n_pad=1, decay_is_log=True)
    pool = w.state_pool()
    hint = max(lengths)
    o1, s1 = _run_fwd(w, pool, max_row_len=hint)
    o0, s0 = _run_fwd(w, pool, max_row_len=0)
    assert (o1.view(np.uint32) == o0.view(np.uint32)).all()
    assert (s1 == s0).all()
    rsi = torch.arange(w.batch, dtype=torch.int32, device=DEV)
    rings, outs, pools = [], [], []
    for h in (hint, 0):
        d = Dev(w, pool)
        ring = ring_for(w, 8, w.batch)
        outs.append(d.verify(ring, rsi, max_row_len=h).cpu().numpy())
        rings.append(ring.cpu().numpy())
        pools.append(pool_to_host(d.state))
    assert (outs[0].view(np.uint32) == outs[1].view(np.uint32)).all()
    assert (np.isnan(rings[0]) == np.isnan(rings[1])).all()
    m = ~np.isnan(rings[0])
    assert (rings[0][m].view(np.uint32) == rings[1][m].view(np.uint32)).all()
    assert (pools[0] == pools[1]).all()
    inters, pools = [], []
    tdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
    for h in (hint, 0):
        d = Dev(w, pool)
        inter = torch.zeros((w.max_slots, 6, w.nv, w.K, w.V), dtype=tdt, device=DEV)
        d.snapshots(inter, 3, max_row_len=h)
        inters.append(pool_to_host(inter))
        pools.append(pool_to_host(d.state))
    assert (inters[0] == inters[1]).all()
    assert (pools[0] == pools[1]).all()
    st = gdr.gdr_get_status(clear=True)
    assert st == 0, gdr.status_names(st)  # the 20-token row has exactly n_inter = 6 drafts of 3


@pytest.mark.parametrize("ring_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [16, 32, 64, 128])
@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
def test_sliced_fold_equals_simple_fold(state_dtype, K, ring_dtype):
    """A 16-byte-aligned ring takes the row-slice fold (where the head size
    allows it), a view offset by one element takes the simple one: same bits."""
    kw = {} if K == 128 else dict(nk=2, nv=6, K=K)
    w = W.verify_fold(batch=40, max_slots=64, ring_rows=64, state_dtype=state_dtype, **kw)
    pool = w.state_pool()
    d = Dev(w, pool)
    ring = ring_for(w, w.ring_len, w.ring_rows, ring_dtype)
    rsi = torch.from_numpy(w.ring_slot_idx).to(DEV)
    d.verify(ring, rsi, max_row_len=12)
    cnt = torch.from_numpy(w.counts).to(DEV)
    outs = []
    for shifted in (False, True):
        st = pool_to_dev(pool_to_host(d.state))
        if shifted:
            buf = torch.empty(ring.numel() + 1, dtype=ring_dtype, device=DEV)
            buf[1:] = ring.reshape(-1)
            r = buf[1:].view(ring.shape)
        else:
            r = ring
        gdr.gdr_fold(st, d.slot, r, rsi, cnt)
        torch.cuda.synchronize()
        outs.append(pool_to_host(st))
    assert (outs[0] == outs[1]).all()
    assert gdr.gdr_get_status(clear=True) == 0


@pytest.mark.parametrize("case", ["decode", "ragged"])
@pytest.mark.parametrize("chunks", [1, 3, 0])
def test_host_buffer_forward_equals_device_forward(case, chunks):
    """gdr_fwd_host (tokens copied in, row groups pipelined over three streams,
    output copied back inside one C-ABI call) gives gdr_fwd's bits: outputs,
    padding zeros and the pool."""
    if case == "decode":
        w = W.decode(batch=40, max_slots=64, n_pad=3)
        mrl = 1
    else:
        w = W.random_case(91, [7, 1, 0, 12, 3, 5, 9], nk=2, nv=4, K=64, max_slots=12,
                          state_dtype="bf16", n_pad=1)
        mrl = 0
    pool = w.state_pool()
    out_ref, pool_ref = _run_fwd(w, pool, max_row_len=mrl)
    state = pool_to_dev(pool)
    hf = gdr.HostForward(state, w.nk, w.batch, w.total_tokens, decay_is_log=w.decay_is_log,
                         use_qk_l2norm=w.use_l2norm, scale=w.scale, eps=w.eps, max_row_len=mrl,
                         chunks=chunks)
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    host_out = torch.full((w.total_tokens, w.nv * w.V), float("nan")).pin_memory()
    hf(pin(w.qkv), pin(w.decay), pin(w.beta), pin(w.slot_idx), pin(w.offsets), host_out)
    torch.cuda.synchronize()
    assert (host_out.numpy().view(np.uint32) == out_ref.view(np.uint32)).all()
    assert (pool_to_host(state) == pool_ref).all()
    assert gdr.gdr_get_status() == 0


def test_longest_first_block_order_does_not_change_bits():
    """Batches of a few rows are dealt to the SMs longest row first (more blocks
    than SMs); a row's bits must not depend on that order: reversing the rows
    of the batch, or running a row alone, gives the same outputs and states."""
    lengths = [37, 300, 5, 181, 96, 250, 64, 141]
    w = W.random_case(612, lengths, nk=16, nv=32, K=128, max_slots=16, state_dtype="bf16")
    pool = w.state_pool()
    out, st = _run_fwd(w, pool)
    rev = sub_workload(w, list(range(w.batch))[::-1])
    out_r, st_r = _run_fwd(rev, pool)
    for i, b in enumerate(range(w.batch)[::-1]):
        t0, t1 = int(w.offsets[b]), int(w.offsets[b + 1])
        r0, r1 = int(rev.offsets[i]), int(rev.offsets[i + 1])
        assert (out_r[r0:r1].view(np.uint32) == out[t0:t1].view(np.uint32)).all(), b
        s = int(w.slot_idx[b])
        assert (st_r[s] == st[s]).all(), b
    for b in (1, 2):
        o, s1 = _run_fwd(sub_workload(w, [b]), pool)
        t0, t1 = int(w.offsets[b]), int(w.offsets[b + 1])
        assert (o.view(np.uint32) == out[t0:t1].view(np.uint32)).all()
        assert (s1[w.slot_idx[b]] == st[w.slot_idx[b]]).all()


def test_host_buffer_forward_single_stream_and_pageable_memory():
    """gdr_fwd_host through the C ABI with no side streams (everything on one
    stream) and with pageable (not pinned) host buffers: the same bits as
    gdr_fwd, and a batch with an empty group of rows."""
    w = W.random_case(93, [0, 4, 0, 0, 6, 2, 0, 9], nk=2, nv=4, K=32, max_slots=10,
                      state_dtype="f32", n_pad=1)
    pool = w.state_pool()
    out_ref, pool_ref = _run_fwd(w, pool)
    state = pool_to_dev(pool)
    hf = gdr.HostForward(state, w.nk, w.batch, w.total_tokens, decay_is_log=w.decay_is_log,
                         use_qk_l2norm=w.use_l2norm, scale=w.scale, eps=w.eps)
    lib = gdr.load_library()
    host = {k: torch.from_numpy(np.ascontiguousarray(v)) for k, v in
            (("qkv", w.qkv), ("decay", w.decay), ("beta", w.beta), ("slot", w.slot_idx),
             ("off", w.offsets))}
    out = torch.full((w.total_tokens, w.nv * w.V), float("nan"))
    io = B.gdr_host_io(host["qkv"].data_ptr(), host["decay"].data_ptr(), host["beta"].data_ptr(),
                       host["slot"].data_ptr(), host["off"].data_ptr(), out.data_ptr())
    stream = torch.cuda.current_stream(DEV).cuda_stream
    for chunks in (5, 1):
        out.fill_(float("nan"))
        state.copy_(pool_to_dev(pool))
        assert lib.gdr_fwd_host(ctypes.byref(hf.args), ctypes.byref(io), chunks, stream, None, None) == 0
        torch.cuda.synchronize()
        assert (out.numpy().view(np.uint32) == out_ref.view(np.uint32)).all(), chunks
        assert (pool_to_host(state) == pool_ref).all(), chunks
    assert gdr.gdr_get_status() == 0
