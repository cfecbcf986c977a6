"""Pins for the oracle's Pass-1 causal depthwise convolution (the producer of
"qkv_conv_output", "gated_delta_recurrence_fwd_gpu" Args): an identity
filter, numpy's correlate on each channel, the impulse response, chaining
through the conv state, short, empty and padding rows, and the SiLU
identity.  None re-types the oracle's loops."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gated_deltanet_linear_gdr_gb300 import workloads as W
from tests.helpers import problem


def _case(seed, lengths, C=6, width=4, slots=5, pad=()):
    rng = np.random.default_rng(seed)
    L = np.asarray(lengths)
    off = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    T = int(off[-1])
    x = rng.standard_normal((T, C)).astype(np.float32)
    w = rng.standard_normal((C, width)).astype(np.float32) * np.float32(0.5)
    bias = rng.standard_normal(C).astype(np.float32) * np.float32(0.1)
    state = rng.standard_normal((slots, C, width - 1)).astype(np.float32)
    slot = rng.permutation(slots)[:len(L)].astype(np.int32)
    for b in pad:
        slot[b] = -1
    return x, w, bias, state, slot, off


def _brute(x, w, bias, silu, state, slot, off):
    """Per channel: numpy's correlate of (state ++ row inputs) with the taps."""
    C, Wd = w.shape
    y = np.zeros(x.shape, np.float64)
    new = state.astype(np.float64).copy()
    for b in range(len(slot)):
        s, t0, t1 = int(slot[b]), int(off[b]), int(off[b + 1])
        if s < 0 or t1 == t0:
            continue
        for c in range(C):
            xe = np.concatenate([state[s, c].astype(np.float64), x[t0:t1, c].astype(np.float64)])
            r = np.correlate(xe, w[c].astype(np.float64), mode="valid")
            if bias is not None:
                r = r + float(bias[c])
            if silu:
                r = r / (1.0 + np.exp(-r))
            y[t0:t1, c] = r
            new[s, c] = xe[len(xe) - (Wd - 1):] if Wd > 1 else []
    return y, new


def test_width_one_identity_filter_returns_the_input():
    x, _, _, _, slot, off = _case(1, [5, 0, 3], width=1)
    w = np.ones((x.shape[1], 1), np.float32)
    y = oracle.conv1d(x, w, None, False, None, slot, off)
    assert (y == x).all()


@pytest.mark.parametrize("silu", [False, True])
@pytest.mark.parametrize("width", [2, 3, 4])
def test_matches_numpy_correlate_per_channel(silu, width):
    x, w, bias, state, slot, off = _case(2 + width, [7, 1, 2, 12, 0], width=width, pad=[1])
    st = state.copy()
    y = oracle.conv1d(x, w, bias, silu, st, slot, off)
    ref, new = _brute(x, w, bias, silu, state, slot, off)
    assert np.abs(y - ref).max() <= 4e-7 * max(1.0, np.abs(ref).max())
    assert (st == new.astype(np.float32)).all()
    assert (y[7:8] == 0).all()  # the padding row's output


def test_impulse_response_is_the_taps_reversed():
    C, Wd, L = 3, 4, 9
    x = np.zeros((L, C), np.float32)
    j0, c0 = 2, 1
    x[j0, c0] = 1.0
    w = np.arange(1, C * Wd + 1, dtype=np.float32).reshape(C, Wd)
    st = np.zeros((1, C, Wd - 1), np.float32)
    y = oracle.conv1d(x, w, None, False, st, np.array([0], np.int32), np.array([0, L], np.int32))
    want = np.zeros((L, C), np.float32)
    for d in range(Wd):
        want[j0 + d, c0] = w[c0, Wd - 1 - d]
    assert (y == want).all()
    # the state keeps the last three inputs
    assert (st[0] == x[L - 3:].T).all()


@pytest.mark.parametrize("cut", [1, 2, 3, 5])
def test_two_calls_chain_through_the_state(cut):
    x, w, bias, state, slot, off = _case(9, [11], width=4)
    st_one = state.copy()
    y_one = oracle.conv1d(x, w, bias, True, st_one, slot, off)
    st_two = state.copy()
    y_a = oracle.conv1d(x[:cut], w, bias, True, st_two, slot, np.array([0, cut], np.int32))
    y_b = oracle.conv1d(x[cut:], w, bias, True, st_two, slot, np.array([0, 11 - cut], np.int32))
    assert (np.concatenate([y_a, y_b]) == y_one).all()
    assert (st_two == st_one).all()


def test_short_row_keeps_part_of_the_old_state():
    x, w, bias, state, slot, off = _case(10, [1, 2], width=4)
    st = state.copy()
    oracle.conv1d(x, w, bias, False, st, slot, off)
    s0, s1 = int(slot[0]), int(slot[1])
    # row 0 (one token): old[1:] then x[0]; row 1 (two tokens): old[2:] then x[1:3]
    assert (st[s0][:, :2] == state[s0][:, 1:]).all() and (st[s0][:, 2] == x[0]).all()
    assert (st[s1][:, 0] == state[s1][:, 2]).all() and (st[s1][:, 1:] == x[1:3].T).all()


def test_padding_and_empty_rows_leave_their_slots():
    x, w, bias, state, slot, off = _case(11, [4, 0, 3], width=4, pad=[2])
    st = state.copy()
    oracle.conv1d(x, w, bias, True, st, slot, off)
    for b in (1, 2):
        s = int(slot[b])
        if s >= 0:
            assert (st[s] == state[s]).all()
    untouched = [s for s in range(state.shape[0]) if s not in set(int(v) for v in slot)]
    assert (st[untouched] == state[untouched]).all()


def test_silu_odd_part_is_the_identity():
    # silu(z) - silu(-z) = z (sigma(z) + sigma(-z) = 1): one tap of weight 1
    z = np.linspace(-6, 6, 25, dtype=np.float32)[:, None]
    w = np.ones((1, 1), np.float32)
    yp = oracle.conv1d(z, w, None, True, None, np.array([0], np.int32), np.array([0, 25], np.int32))
    yn = oracle.conv1d(-z, w, None, True, None, np.array([0], np.int32), np.array([0, 25], np.int32))
    assert np.abs(yp.astype(np.float64) - yn - z).max() <= 1e-6
    assert yp[12, 0] == 0.0


def test_forward_on_conv_output_equals_forward_on_its_input_for_the_identity_filter():
    w = W.random_case(12, [6, 0, 3], nk=1, nv=2, K=16, max_slots=4, state_dtype="f32")
    C = w.qkv.shape[1]
    p1 = problem(w, state=w.state_pool())
    ref = oracle.fwd(p1)
    p2 = problem(w, state=w.state_pool())
    out = oracle.fwd_conv(p2, np.ones((C, 1), np.float32), None, False, None)
    assert (out == ref).all()
    assert (p2.state == p1.state).all()
