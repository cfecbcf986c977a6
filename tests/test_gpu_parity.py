"""GPU path vs the CPU oracle on the same seeded inputs, through the C ABI.

Tolerances: outputs max abs 2e-3; bf16 state within one bf16 ulp of the
oracle (floor 2^-10); float32 state, ring and snapshots 1e-4 abs/rel; slot,
record and snapshot bookkeeping exact."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import gated_deltanet_linear_gdr_gb300 as gdr
from gated_deltanet_linear_gdr_gb300 import workloads as W
from tests.gpu_helpers import (DEV, Dev, as_f64, check_out, check_state, pool_to_dev, pool_to_host,
                               ring_for, ring_to_dev, ring_to_host)
from tests.helpers import problem, sub_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    gdr.gdr_get_status(clear=True)
    yield
    st = gdr.gdr_get_status(clear=True)
    assert st == 0, f"device status {gdr.status_names(st)}"


def _fwd_parity(w, max_row_len=0):
    pool = w.state_pool()
    d = Dev(w, pool)
    out = d.fwd(max_row_len=max_row_len)
    torch.cuda.synchronize()
    p = problem(w, state=pool.copy())
    ref = oracle.fwd(p)
    check_out(out, ref)
    check_state(pool_to_host(d.state), p.state)
    return out, d, p


def test_tiny_config():
    _fwd_parity(W.tiny())


@pytest.mark.parametrize("K", [16, 32, 64, 128])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hint", [0, 40])  # 0: general kernel; 40: short-row kernel where it applies
def test_ragged_rows_all_head_dims(K, state_dtype, hint):
    # lengths span several staged chunks (8 and 16 tokens) with ragged tails, plus
    # empty and single-token rows and a padding row; GQA ratio 2
    lengths = [37, 0, 1, 16, 5, 33]
    w = W.random_case(100 + K, lengths, nk=2, nv=4, K=K, max_slots=9, state_dtype=state_dtype,
                      n_pad=1)
    _fwd_parity(w, max_row_len=hint)


@pytest.mark.parametrize("K", [16, 32, 64, 128])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_decode_kernel_all_head_dims(K, state_dtype):
    w = W.random_case(200 + K, [1] * 7 + [0], nk=2, nv=6, K=K, max_slots=12,
                      state_dtype=state_dtype, n_pad=2)
    _fwd_parity(w, max_row_len=1)


@pytest.mark.parametrize("variant", ["no_l2norm", "log_decay", "scale", "gqa4", "mha"])
def test_variants(variant):
    kw = dict(nk=2, nv=4, K=64, max_slots=6, state_dtype="bf16")
    if variant == "no_l2norm":
        w = W.random_case(300, [9, 20], use_l2norm=False, state_std=0.02, **kw)
        # raw q/k are unnormalised: keep the output scale comparable to the tolerance
        w = dataclasses.replace(w, qkv=w.qkv * np.float32(0.125))
    elif variant == "log_decay":
        w = W.random_case(301, [9, 20], decay_is_log=True, **kw)
    elif variant == "scale":
        w = W.random_case(302, [9, 20], scale=0.3, **kw)
    elif variant == "gqa4":
        w = W.random_case(303, [9, 20], **{**kw, "nk": 1})
    else:
        w = W.random_case(304, [9, 20], **{**kw, "nk": 4})
    _fwd_parity(w)
    _fwd_parity(dataclasses.replace(w, offsets=w.offsets), max_row_len=0)


def test_decode_config_full_size():
    """The decode workload exactly as timed: batch 256, one token, 8 padding rows,
    nk=16, nv=32, K=V=128, bf16 pool [512, 32, 128, 128]."""
    w = W.decode()
    out, d, p = _fwd_parity(w, max_row_len=1)
    pad = w.slot_idx < 0
    assert (out.cpu().numpy()[pad] == 0).all()


def test_decode_config_through_general_kernel():
    w = W.decode(batch=64, max_slots=128)
    _fwd_parity(w, max_row_len=0)


def test_prefill_config_sampled_rows():
    """The ragged prefill workload at full size on the GPU; the oracle recomputes
    the two shortest rows, a middle one and the longest (3514 tokens at this
    seed: the row where float32 rounding has the longest run to build up and
    the bf16 state must still land within one ulp).  Rows are independent."""
    w = W.prefill()
    pool = w.state_pool()
    d = Dev(w, pool)
    out = d.fwd()
    torch.cuda.synchronize()
    L = w.row_lengths
    order = np.argsort(L, kind="stable")
    rows = sorted({int(order[0]), int(order[1]), int(order[len(order) // 2]), int(order[-1])})
    assert L[rows].max() == L.max()
    sub = sub_workload(w, rows)
    p = problem(sub, state=pool.copy())
    ref = oracle.fwd(p)
    got = out.cpu().numpy()
    toks = np.concatenate([np.arange(w.offsets[b], w.offsets[b + 1]) for b in rows])
    err = np.abs(got[toks].astype(np.float64) - ref).max()
    assert err <= 2e-3, err
    host = pool_to_host(d.state)
    check_state(host, p.state, slots=[int(w.slot_idx[b]) for b in rows])


@pytest.mark.parametrize("hint", [0, 12])  # 0: general kernel; 12: short-row kernel
def test_verify_fold_config(hint):
    w = W.verify_fold()
    pool = w.state_pool()
    d = Dev(w, pool)
    ring = ring_for(w, w.ring_len, w.ring_rows)
    rsi = torch.from_numpy(w.ring_slot_idx).to(DEV)
    out = d.verify(ring, rsi, max_row_len=hint)
    torch.cuda.synchronize()
    pv = problem(w, state=pool.copy())
    oring = np.full(tuple(ring.shape), np.nan, np.float32)
    ref = oracle.verify_ring(pv, oring, w.ring_slot_idx, w.ring_len)
    check_out(out, ref)
    host = pool_to_host(d.state)
    long_rows = [b for b in range(w.batch) if w.row_lengths[b] > w.ring_len]
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        if b in long_rows:
            check_state(host, pv.state, slots=[s])
        else:
            assert (host[s] == pool[s]).all(), "verify wrote the pool"
    # records: same fields written, values within float32 tolerance
    g = ring.cpu().numpy()
    assert (np.isnan(g) == np.isnan(oring)).all()
    m = ~np.isnan(oring)
    np.testing.assert_allclose(g[m], oring[m], rtol=1e-4, atol=1e-4)
    # fold with the accepted counts, against the oracle's fold of its own records
    cnt = torch.from_numpy(w.counts).to(DEV)
    gdr.gdr_fold(d.state, d.slot, ring, rsi, cnt)
    torch.cuda.synchronize()
    oracle.fold(pv, oring, w.ring_slot_idx, w.counts, w.ring_len)
    check_state(pool_to_host(d.state), pv.state, slots=w.live_slots())


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_fold_on_synthetic_ring(state_dtype):
    """Fold alone on a random ring (not produced by any verify pass)."""
    nk, nv, K, ring_len = 2, 4, 128, 8
    w = W.random_case(400, [1] * 6, nk=nk, nv=nv, K=K, max_slots=10, state_dtype=state_dtype)
    w = dataclasses.replace(w, slot_idx=np.array([3, -1, 7, 0, 9, 5], np.int32))
    stride = gdr.gdr_ring_record_elements(K, K, nv // nk)
    rng = np.random.default_rng(401)
    ring = (rng.standard_normal((6, nk, ring_len, stride)) * 0.3).astype(np.float32)
    ring[..., K:K + 4] = rng.uniform(0.8, 1.0, (6, nk, ring_len, 4)).astype(np.float32)
    rsi = np.array([5, 4, 3, 2, 1, 0], np.int32)
    counts = np.array([3, 2, 0, 8, 9, 1], np.int32)
    pool = w.state_pool()
    st = pool_to_dev(pool)
    gdr.gdr_fold(st, torch.from_numpy(w.slot_idx).to(DEV), torch.from_numpy(ring).to(DEV),
                 torch.from_numpy(rsi).to(DEV), torch.from_numpy(counts).to(DEV))
    torch.cuda.synchronize()
    p = problem(w, state=pool.copy())
    oracle.fold(p, ring, rsi, counts, ring_len)
    host = pool_to_host(st)
    check_state(host, p.state)
    for b, s in enumerate(w.slot_idx):
        if s >= 0 and (counts[b] == 0 or counts[b] > ring_len):
            assert (host[s] == pool[s]).all()


@pytest.mark.parametrize("K", [16, 64, 128])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hint", [0, 1])
def test_value_head_twice_key_head_forward(K, state_dtype, hint):
    """V = 2K ("core.ssm.ops.gdp.fused_recurrent": K and V sized separately)
    against the oracle, ragged rows with a padding row."""
    lengths = [1, 18, 0, 7] if hint == 0 else [1, 1, 1, 0]
    w = W.random_case(800 + K, lengths, nk=2, nv=4, K=K, V=2 * K, max_slots=9, state_dtype=state_dtype,
                      n_pad=1)
    _fwd_parity(w, max_row_len=hint)


@pytest.mark.parametrize("K", [32, 64, 128])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hint", [0, 1, 16])  # the general kernel's 32-, 8- and 16-token chunks
def test_key_head_twice_value_head_forward(K, state_dtype, hint):
    """V = K/2 ("core.ssm.ops.gdp.fused_recurrent": q, k [B, T, H, K] and v
    [B, T, HV, V] sized separately) against the oracle: ragged rows, an empty
    row and a padding row."""
    lengths = [1, 18, 0, 7, 40] if hint == 0 else [1, 1, 1, 0] if hint == 1 else [16, 3, 0, 9]
    w = W.random_case(830 + K + hint, lengths, nk=2, nv=4, K=K, V=K // 2, max_slots=9,
                      state_dtype=state_dtype, n_pad=1)
    _fwd_parity(w, max_row_len=hint)


@pytest.mark.parametrize("K", [32, 128])
def test_key_head_twice_value_head_beta_per_value(K):
    w = W.random_case(850 + K, [5, 12, 1], nk=1, nv=2, K=K, V=K // 2, max_slots=4, state_dtype="bf16",
                      beta_per_value=True)
    _fwd_parity(w)


@pytest.mark.parametrize("V", [128, 32])  # 2K and K/2
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_value_head_twice_key_head_snapshots_rollback_dense(state_dtype, V):
    w = W.random_case(810, [8, 6, 8], nk=2, nv=4, K=64, V=V, max_slots=6, state_dtype=state_dtype,
                      decay_is_log=True)
    pool = w.state_pool()
    d = Dev(w, pool)
    tdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
    inter = torch.zeros((w.max_slots, 4, w.nv, w.K, w.V), dtype=tdt, device=DEV)
    out = d.snapshots(inter, 2)
    torch.cuda.synchronize()
    p = problem(w, state=pool.copy())
    oint = np.zeros(tuple(inter.shape), pool.dtype)
    ref = oracle.fwd_snapshots(p, oint, 2)
    check_out(out, ref)
    check_state(pool_to_host(inter), oint)
    check_state(pool_to_host(d.state), p.state)
    acc = np.array([1, 2, 3], np.int32)
    gdr.gdr_rollback(d.state, d.slot, inter, torch.from_numpy(acc).to(DEV))
    oracle.rollback(p, oint, acc)
    torch.cuda.synchronize()
    check_state(pool_to_host(d.state), p.state)
    # dense start state, V = 2K
    kw = dict(nk=w.nk, nv=w.nv, K=w.K, V=w.V, state_dtype=state_dtype, decay_is_log=True,
              use_l2norm=w.use_l2norm, scale=w.scale, eps=w.eps)
    init = pool[w.slot_idx]
    ref_out, ref_final = oracle.fwd_dense(w.qkv, w.decay, w.beta, w.offsets, init, **kw)
    out_d, final = gdr.gdr_fwd_dense(d.qkv, d.decay, d.beta, d.off, pool_to_dev(init), decay_is_log=True)
    torch.cuda.synchronize()
    check_out(out_d, ref_out)
    check_state(pool_to_host(final), ref_final)


@pytest.mark.parametrize("K", [16, 64, 128])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("with_initial", [True, False])
def test_dense_state_forward(K, state_dtype, with_initial):
    """initial_state / output_final_state ("core.ssm.ops.gdp.fused_recurrent")
    against the oracle: ragged rows, an empty row (its final state is its start
    state), with and without a start state."""
    w = W.random_case(700 + K, [21, 0, 5, 1], nk=2, nv=4, K=K, max_slots=4, state_dtype=state_dtype)
    init = w.state_pool()[np.arange(w.batch)] if with_initial else None
    kw = dict(nk=w.nk, nv=w.nv, K=w.K, V=w.V, state_dtype=state_dtype, decay_is_log=w.decay_is_log,
              use_l2norm=w.use_l2norm, scale=w.scale, eps=w.eps)
    ref_out, ref_final = oracle.fwd_dense(w.qkv, w.decay, w.beta, w.offsets, init, **kw)
    tdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
    out, final = gdr.gdr_fwd_dense(
        torch.from_numpy(w.qkv).to(DEV), torch.from_numpy(w.decay).to(DEV),
        torch.from_numpy(w.beta).to(DEV), torch.from_numpy(w.offsets).to(DEV),
        None if init is None else pool_to_dev(init), nv=w.nv, K=w.K, state_dtype=tdt)
    torch.cuda.synchronize()
    check_out(out, ref_out)
    check_state(pool_to_host(final), ref_final)
    if init is not None:
        assert (pool_to_host(final)[1] == init[1]).all(), "an empty row hands its start state on"
    else:
        assert (as_f64(pool_to_host(final)[1]) == 0).all()


@pytest.mark.parametrize("K", [16, 32, 64, 128])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hint", [0, 1, 40])
def test_beta_per_value_forward(K, state_dtype, hint):
    """beta [T, HV, V] ("core.ssm.ops.gdp.fused_recurrent" Parameters) against
    the oracle; ragged rows over several staged chunks, a padding row, every
    kernel hint (per-element beta always runs on the general kernel)."""
    lengths = [1, 19, 0, 9] if hint != 1 else [1, 1, 0, 1]
    w = W.random_case(600 + K, lengths, nk=2, nv=4, K=K, max_slots=9, state_dtype=state_dtype,
                      n_pad=1, beta_per_value=True)
    _fwd_parity(w, max_row_len=hint)


def test_beta_per_value_strided_and_snapshots():
    """A non-contiguous per-element beta (scalar staging) and the snapshot pass."""
    w = W.random_case(610, [8, 6, 8], nk=2, nv=4, K=64, max_slots=6, state_dtype="f32",
                      beta_per_value=True, decay_is_log=True)
    pool = w.state_pool()
    d = Dev(w, pool)
    bt = torch.from_numpy(np.ascontiguousarray(w.beta.transpose(2, 0, 1))).to(DEV)  # [V, T, nv]
    d.beta = bt.permute(1, 2, 0)  # [T, nv, V] view with value-dim stride T*nv
    inter = torch.full((w.max_slots, 4, w.nv, w.K, w.V), float("nan"), device=DEV)
    out = d.snapshots(inter, 2)
    torch.cuda.synchronize()
    p = problem(w, state=pool.copy())
    oint = np.full((w.max_slots, 4, w.nv, w.K, w.V), np.nan, np.float32)
    ref = oracle.fwd_snapshots(p, oint, 2)
    check_out(out, ref)
    hi = inter.cpu().numpy()
    written = ~np.isnan(oint)
    assert (written == ~np.isnan(hi)).all(), "snapshot entries written where the oracle writes"
    hi[~written] = 0.0
    oint[~written] = 0.0
    check_state(hi, oint)
    check_state(pool_to_host(d.state), p.state)


@pytest.mark.parametrize("hint", [0, 12])  # 0: general kernel; 12: short-row kernel
@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
def test_bf16_ring_verify_records_and_fold(state_dtype, hint):
    """bfloat16 ring ("gated_delta_recurrence_verify_ring_gpu" Parameters:
    ring_dtype): verify writes the forward pass's output and records within one
    bfloat16 ulp of the oracle's (each side rounds its own value once); the fold
    of the oracle's bfloat16 records matches the oracle's fold of them."""
    w = W.verify_fold(batch=24, max_slots=48, ring_rows=48, nk=4, nv=8, state_dtype=state_dtype)
    pool = w.state_pool()
    d = Dev(w, pool)
    ring = ring_for(w, w.ring_len, w.ring_rows, torch.bfloat16)
    rsi = torch.from_numpy(w.ring_slot_idx).to(DEV)
    out = d.verify(ring, rsi, max_row_len=hint)
    torch.cuda.synchronize()
    pv = problem(w, state=pool.copy())
    oring = np.full(tuple(ring.shape), 0x7FC0, np.uint16)
    ref = oracle.verify_ring(pv, oring, w.ring_slot_idx, w.ring_len)
    check_out(out, ref)
    g = ring_to_host(ring)
    nan = 0x7FC0
    assert ((g == nan) == (oring == nan)).all(), "same record fields written"
    m = oring != nan
    gf, rf = as_f64(g[m]), as_f64(oring[m])
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(rf), 2.0 ** -20))) - 7)
    bad = np.abs(gf - rf) > ulp * 1.001
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} records beyond one bfloat16 ulp"
    # fold the oracle's records on the GPU and in the oracle
    st = pool_to_dev(pool)
    gdr.gdr_fold(st, d.slot, ring_to_dev(oring), rsi, torch.from_numpy(w.counts).to(DEV))
    torch.cuda.synchronize()
    pf = problem(w, state=pool.copy())
    oracle.fold(pf, oring, w.ring_slot_idx, w.counts, w.ring_len)
    check_state(pool_to_host(st), pf.state, slots=w.live_slots())


@pytest.mark.parametrize("hint", [0, 8])  # 0: general kernel; 8: short-row kernel
def test_gdp_snapshot_config_and_rollback(hint):
    """Gated Delta Product spec-decode at full size: 64 requests x 4 drafts x 2
    Householder copies, fp32 cache [128, 32, 128, 128], snapshots every 2 steps,
    then rollback to a random accepted draft."""
    w = W.gdp_snapshots()
    pool = w.state_pool()
    d = Dev(w, pool)
    inter = torch.full((w.max_slots, w.n_inter, w.nv, w.K, w.V), float("nan"), device=DEV)
    out = d.snapshots(inter, w.steps_per_token, max_row_len=hint)
    torch.cuda.synchronize()
    sub_rows = list(range(w.batch))  # the oracle over every request
    sub = sub_workload(w, sub_rows)
    p = problem(sub, state=pool.copy())
    oint = np.full((w.max_slots, w.n_inter, w.nv, w.K, w.V), np.nan, np.float32)
    ref = oracle.fwd_snapshots(p, oint, w.steps_per_token)
    toks = np.concatenate([np.arange(w.offsets[b], w.offsets[b + 1]) for b in sub_rows])
    err = np.abs(out.cpu().numpy()[toks].astype(np.float64) - ref).max()
    assert err <= 2e-3, err
    slots = [int(w.slot_idx[b]) for b in sub_rows]
    host_inter = inter.cpu().numpy()
    check_state(host_inter, oint, slots=slots)
    check_state(pool_to_host(d.state), p.state, slots=slots)
    # snapshots exist exactly for the live slots
    live = set(w.live_slots())
    for s in range(w.max_slots):
        assert np.isnan(host_inter[s]).all() == (s not in live)
    # rollback
    acc = torch.from_numpy(w.accepted).to(DEV)
    gdr.gdr_rollback(d.state, d.slot, inter, acc)
    torch.cuda.synchronize()
    host = pool_to_host(d.state)
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        assert (host[s] == host_inter[s, w.accepted[b]]).all()


def test_snapshot_small_bf16_against_oracle():
    w = W.random_case(500, [8, 7, 8, 3], nk=2, nv=4, K=32, max_slots=6, state_dtype="bf16",
                      n_pad=1, decay_is_log=True)
    pool = w.state_pool()
    d = Dev(w, pool)
    inter = torch.zeros((w.max_slots, 4, w.nv, w.K, w.V), dtype=torch.bfloat16, device=DEV)
    out = d.snapshots(inter, 2)
    p = problem(w, state=pool.copy())
    oint = np.zeros((w.max_slots, 4, w.nv, w.K, w.V), np.uint16)
    ref = oracle.fwd_snapshots(p, oint, 2)
    check_out(out, ref)
    check_state(pool_to_host(inter), oint)
    check_state(pool_to_host(d.state), p.state)


@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
def test_limits_ring_len_32_and_64_token_rows(state_dtype):
    """The largest ring (RING_LEN 32) with rows of exactly 32 tokens (they
    record) and 33 and 64 (they commit like the forward pass), the latter at
    the short-row kernel's 64-token limit: verify against the oracle through
    both kernels, which agree bit for bit, then fold against the oracle's fold."""
    lengths = [32, 33, 64, 1, 17, 0]
    w = W.random_case(713, lengths, nk=2, nv=4, K=64, max_slots=8, state_dtype=state_dtype, n_pad=0)
    pool = w.state_pool()
    ring_len, rows = 32, w.batch
    rsi_np = np.arange(w.batch, dtype=np.int32)[::-1].copy()
    rsi = torch.from_numpy(rsi_np).to(DEV)
    pv = problem(w, state=pool.copy())
    oring = np.full((rows, w.nk, ring_len, ring_for(w, ring_len, rows).shape[3]), np.nan, np.float32)
    ref = oracle.verify_ring(pv, oring, rsi_np, ring_len)
    got = []
    for hint in (64, 0):
        d = Dev(w, pool)
        ring = ring_for(w, ring_len, rows)
        out = d.verify(ring, rsi, max_row_len=hint)
        torch.cuda.synchronize()
        check_out(out, ref)
        host = pool_to_host(d.state)
        for b, L in enumerate(lengths):
            s = int(w.slot_idx[b])
            if L > ring_len:
                check_state(host, pv.state, slots=[s])
            else:
                assert (host[s] == pool[s]).all(), b
        g = ring.cpu().numpy()
        assert (np.isnan(g) == np.isnan(oring)).all()
        m = ~np.isnan(oring)
        np.testing.assert_allclose(g[m], oring[m], rtol=1e-4, atol=1e-4)
        got.append((out.cpu().numpy(), g, host, d, ring))
    assert (got[0][0].view(np.uint32) == got[1][0].view(np.uint32)).all()
    m = ~np.isnan(got[0][1])
    assert (got[0][1][m].view(np.uint32) == got[1][1][m].view(np.uint32)).all()
    assert (got[0][2] == got[1][2]).all()
    counts = np.array([32, 33, 64, 1, 9, 0], np.int32)
    _, _, _, d, ring = got[0]
    gdr.gdr_fold(d.state, d.slot, ring, rsi, torch.from_numpy(counts).to(DEV))
    torch.cuda.synchronize()
    oracle.fold(pv, oring, rsi_np, counts, ring_len)
    check_state(pool_to_host(d.state), pv.state, slots=w.live_slots())
    assert gdr.gdr_get_status(clear=True) == 0
