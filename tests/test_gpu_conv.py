"""The forward pass with the Pass-1 convolution fused into operand staging
(gdr_fwd_conv; "gated_delta_recurrence_fwd_gpu", Args: qkv_conv_output is
the "Conv1d output from Pass 1") against the oracle's conv1d followed by its
forward pass, through the C ABI.  Tolerances as for the forward pass; the
conv state holds copies of raw inputs and must match exactly."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import gated_deltanet_linear_gdr_gb300 as gdr
from gated_deltanet_linear_gdr_gb300 import workloads as W
from tests.gpu_helpers import DEV, Dev, check_out, check_state, pool_to_host
from tests.helpers import problem, sub_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    gdr.gdr_get_status(clear=True)
    yield
    st = gdr.gdr_get_status(clear=True)
    assert st == 0, f"device status {gdr.status_names(st)}"


def _t(x):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def _gpu_conv(w, pool, cv, max_row_len=0, conv_state=None):
    d = Dev(w, pool)
    cs = _t(cv.state) if conv_state is None else conv_state
    out = gdr.gdr_fwd_conv(d.qkv, d.decay, d.beta, d.state, d.slot, d.off, _t(cv.weight), _t(cv.bias), cs,
                           activation="silu" if cv.silu else None, max_row_len=max_row_len, **d.kw)
    torch.cuda.synchronize()
    return out, d, cs


def _oracle_conv(w, pool, cv):
    p = problem(w, state=pool.copy())
    cs = None if cv.state is None else cv.state.copy()
    ref = oracle.fwd_conv(p, cv.weight, cv.bias, cv.silu, cs)
    return ref, p, cs


@pytest.mark.parametrize("state_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("hint", [0, 8])
def test_identity_filter_equals_the_plain_forward_pass(state_dtype, hint):
    """Width 1, weight 1, no bias, no activation: gdr_fwd's bits."""
    lengths = [5, 0, 1, 8] if hint else [5, 0, 1, 40, 17]
    w = W.random_case(900, lengths, nk=2, nv=4, K=128, max_slots=8, state_dtype=state_dtype, n_pad=1)
    pool = w.state_pool()
    ident = W.ConvInputs(np.ones((w.qkv.shape[1], 1), np.float32), None, None, False)
    out_c, d_c, _ = _gpu_conv(w, pool, ident, max_row_len=hint)
    d = Dev(w, pool)
    out = d.fwd(max_row_len=hint)
    torch.cuda.synchronize()
    assert (out_c.cpu().numpy().view(np.uint32) == out.cpu().numpy().view(np.uint32)).all()
    assert (pool_to_host(d_c.state) == pool_to_host(d.state)).all()


@pytest.mark.parametrize("K", [16, 32, 64, 128])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("width,silu,bias", [(4, True, True), (3, False, True), (2, True, False)])
def test_ragged_rows_against_the_oracle(K, state_dtype, width, silu, bias):
    # rows across several 16-token chunks, rows shorter than the filter, an
    # empty row and a padding row
    lengths = [37, 0, 1, 2, 16, 5]
    w = W.random_case(910 + K + width, lengths, nk=2, nv=4, K=K, max_slots=9, state_dtype=state_dtype, n_pad=1)
    pool = w.state_pool()
    cv = W.conv_inputs(w, width=width, seed=K, bias=bias, silu=silu)
    out, d, cs = _gpu_conv(w, pool, cv)
    ref, p, cs_ref = _oracle_conv(w, pool, cv)
    check_out(out, ref)
    check_state(pool_to_host(d.state), p.state)
    assert (cs.cpu().numpy() == cs_ref).all(), "conv state"


def test_short_row_chunks_against_the_oracle():
    w = W.random_case(920, [8, 3, 1, 7], nk=1, nv=2, K=64, max_slots=6, state_dtype="bf16")
    pool = w.state_pool()
    cv = W.conv_inputs(w, width=4, seed=3)
    out, d, cs = _gpu_conv(w, pool, cv, max_row_len=8)
    ref, p, cs_ref = _oracle_conv(w, pool, cv)
    check_out(out, ref)
    check_state(pool_to_host(d.state), p.state)
    assert (cs.cpu().numpy() == cs_ref).all()


def test_decode_config_full_size():
    """The decode workload (256 rows x 1 token, 8 padding rows, nk=16, nv=32,
    K=V=128, bf16 pool) through the fused convolution, width 4, SiLU, bias,
    conv state [512, 8192, 3]."""
    w = W.decode()
    pool = w.state_pool()
    cv = W.conv_inputs(w, width=4, seed=1)
    out, d, cs = _gpu_conv(w, pool, cv, max_row_len=1)
    ref, p, cs_ref = _oracle_conv(w, pool, cv)
    check_out(out, ref)
    check_state(pool_to_host(d.state), p.state, slots=w.live_slots())
    assert (cs.cpu().numpy() == cs_ref).all()
    assert (out.cpu().numpy()[w.slot_idx < 0] == 0).all()


def test_prefill_config_sampled_rows():
    """The ragged prefill workload (8 rows, T = 15 843) through the fused
    convolution; the oracle recomputes the shortest, a middle and the longest
    row (rows are independent), and every row's conv state."""
    w = W.prefill()
    pool = w.state_pool()
    cv = W.conv_inputs(w, width=4, seed=2)
    out, d, cs = _gpu_conv(w, pool, cv)
    L = w.row_lengths
    order = np.argsort(L, kind="stable")
    rows = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    sub = sub_workload(w, rows)
    ref, p, _ = _oracle_conv(sub, pool, cv)
    toks = np.concatenate([np.arange(w.offsets[b], w.offsets[b + 1]) for b in rows])
    err = np.abs(out.cpu().numpy()[toks].astype(np.float64) - ref).max()
    assert err <= 2e-3, err
    check_state(pool_to_host(d.state), p.state, slots=[int(w.slot_idx[b]) for b in rows])
    # conv state of every row: the last three raw inputs
    got = cs.cpu().numpy()
    for b in range(w.batch):
        s, t1 = int(w.slot_idx[b]), int(w.offsets[b + 1])
        assert (got[s] == w.qkv[t1 - 3:t1].T).all(), b


def test_two_calls_chain_through_both_states():
    """float32 pool: one call over a row == two calls over its halves, the
    recurrence state and the conv state carried between them, bit for bit."""
    w = W.random_case(930, [23, 40, 2], nk=2, nv=4, K=64, max_slots=5, state_dtype="f32")
    pool = w.state_pool()
    cv = W.conv_inputs(w, width=4, seed=5)
    out, d, cs = _gpu_conv(w, pool, cv)
    cuts = [10, 17, 1]
    st, cs2 = pool.copy(), _t(cv.state)
    outs = []
    for first in (True, False):
        rows = []
        for b in range(w.batch):
            t0, t1 = int(w.offsets[b]), int(w.offsets[b + 1])
            c = t0 + cuts[b]
            rows.append((t0, c) if first else (c, t1))
        toks = np.concatenate([np.arange(a, z) for a, z in rows])
        offs = np.concatenate([[0], np.cumsum([z - a for a, z in rows])]).astype(np.int32)
        part = dataclasses.replace(w, qkv=w.qkv[toks], decay=w.decay[toks], beta=w.beta[toks], offsets=offs)
        o, dd, cs2 = _gpu_conv(part, st, cv, conv_state=cs2)
        st = pool_to_host(dd.state)
        outs.append((o.cpu().numpy(), toks))
    assert (st == pool_to_host(d.state)).all()
    assert (cs2.cpu().numpy() == cs.cpu().numpy()).all()
    full = out.cpu().numpy()
    for o, toks in outs:
        assert (o.view(np.uint32) == full[toks].view(np.uint32)).all()


def test_skipped_rows_keep_their_conv_state():
    """A padding row and a row longer than max_row_len leave their conv state
    alone (the longer row is flagged and its output zeroed)."""
    w = W.random_case(940, [3, 2, 9], nk=1, nv=2, K=32, max_slots=5, state_dtype="f32")
    w = dataclasses.replace(w, slot_idx=np.array([1, -1, 3], np.int32))
    pool = w.state_pool()
    cv = W.conv_inputs(w, width=4, seed=6)
    out, d, cs = _gpu_conv(w, pool, cv, max_row_len=8)
    st = gdr.gdr_get_status(clear=True)
    assert st == 0x10, gdr.status_names(st)
    got = cs.cpu().numpy()
    assert (got[3] == cv.state[3]).all() and (got[[0, 2, 4]] == cv.state[[0, 2, 4]]).all()
    assert (got[1] == w.qkv[0:3].T).all()
    assert (out.cpu().numpy()[3:] == 0).all()


def test_binding_rejects_a_conv_state_smaller_than_the_pool():
    w = W.random_case(950, [3], nk=1, nv=2, K=16, max_slots=4, state_dtype="f32")
    d = Dev(w, w.state_pool())
    cv = W.conv_inputs(w, width=4)
    with pytest.raises(ValueError, match="one row per pool slot"):
        gdr.gdr_fwd_conv(d.qkv, d.decay, d.beta, d.state, d.slot, d.off, _t(cv.weight), _t(cv.bias),
                         _t(cv.state[:3]), **d.kw)
