"""Pins for the CPU oracle: closed forms, invariants, brute force and exact
arithmetic.  None of these re-types the oracle's loops; each checks it against
something the pages or the mathematics fix independently."""
from __future__ import annotations

import dataclasses
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import brute, exact
from gated_deltanet_linear_gdr_gb300 import workloads as W
from tests.helpers import problem, state_f64, sub_workload


# ---------------------------------------------------------------- storage ---

def test_bf16_rounding_matches_torch_on_float32_inputs():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(123)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(0.05),
        rng.standard_normal(1000).astype(np.float32) * np.float32(1e30),
        (rng.standard_normal(500) * 1e-39).astype(np.float32),  # float32 subnormals
        np.array([0.0, -0.0, 1.0, -1.0, 3.4e38, -3.4e38], dtype=np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(x.astype(np.float64))
    assert (got == want).all()


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0).
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even).
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above the tie rounds up
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    # largest finite and overflow
    assert oracle.round_bf16(255 * 2.0 ** 120) == 0x7F7F
    assert oracle.round_bf16(2.0 ** 128 - 2.0 ** 119) == 0x7F80
    # double-only precision: a value that double rounding (f64->f32->bf16) gets wrong
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40  # f32 rounds this to exactly the tie 1+2^-8
    assert oracle.round_bf16(x) == 0x3F81
    assert (oracle.bf16_to_f64(np.array([0x3F81], dtype=np.uint16)) == 1.0 + 2.0 ** -7).all()


def test_ring_record_elements():
    # [k^ (K) | alpha x r padded to 8 | u x r (V each)]
    assert oracle.ring_record_elements(128, 128, 2) == 128 + 8 + 256
    assert oracle.ring_record_elements(16, 16, 1) == 16 + 8 + 16
    assert oracle.ring_record_elements(64, 64, 9) == 64 + 16 + 576


# ------------------------------------------------------ brute-force pins ---

def _small(seed, lengths, nk, nv, K, **kw):
    return W.random_case(seed, lengths, nk, nv, K, max_slots=len(lengths) + 3, **kw)


@pytest.mark.parametrize("use_l2norm", [True, False])
@pytest.mark.parametrize("decay_is_log", [False, True])
def test_matches_matrix_form_bruteforce(use_l2norm, decay_is_log):
    w = _small(11, [3, 0, 5, 1], nk=2, nv=4, K=4, n_pad=1, use_l2norm=use_l2norm,
               decay_is_log=decay_is_log, scale=0.0, state_dtype="f32")
    pool = w.state_pool(w.live_slots())
    ref_out, finals = brute.fwd(w.qkv, w.decay, w.beta, pool, w.slot_idx, w.offsets,
                                nk=w.nk, nv=w.nv, K=w.K, V=w.V, decay_is_log=decay_is_log,
                                use_l2norm=use_l2norm)
    p = problem(w, state=pool.copy())
    out = oracle.fwd(p)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    for (slot, h), S in finals.items():
        # the pool stores float32: compare against the float32 rounding of the exact state
        np.testing.assert_array_equal(p.state[slot, h], S.astype(np.float32))


@pytest.mark.parametrize("KV", [(4, 8), (8, 4)])
def test_matches_matrix_form_bruteforce_k_ne_v(KV):
    """K != V ("core.ssm.ops.gdp.fused_recurrent": K and V are separate sizes)."""
    K, V = KV
    w = _small(14, [3, 4], nk=1, nv=2, K=K, V=V)
    pool = w.state_pool()
    p = problem(w, state=pool.copy())
    out = oracle.fwd(p)
    ref_out, finals = brute.fwd(w.qkv, w.decay, w.beta, pool, w.slot_idx, w.offsets,
                                nk=w.nk, nv=w.nv, K=K, V=V, eps=w.eps)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-12)
    for (s, h), S in finals.items():
        np.testing.assert_allclose(p.state[s, h], S, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("seed", range(16))
def test_random_shapes_match_matrix_form_bruteforce(seed):
    """A sweep over small random shapes and options: key/value head counts with
    GQA groups of 1, 2 or 4, K from 2 to 16, V = K or 2K, ragged row lengths
    including empty rows, padding rows, either decay form, with or without the
    L2 norm, default or explicit scale.  Each draw is checked against the
    matrix-form step ("core.ssm.ops.gdp.fused_recurrent")."""
    rng = np.random.default_rng(1000 + seed)
    nk = int(rng.choice([1, 2]))
    nv = nk * int(rng.choice([1, 2, 4]))
    K = int(rng.choice([2, 4, 8, 16]))
    V = K * int(rng.choice([1, 2]))
    lengths = [int(x) for x in rng.integers(0, 7, size=int(rng.integers(1, 6)))]
    n_pad = int(rng.integers(0, len(lengths)))
    log = bool(rng.integers(0, 2))
    l2 = bool(rng.integers(0, 2))
    scale = float(rng.choice([0.0, 0.37]))
    w = _small(2000 + seed, lengths, nk=nk, nv=nv, K=K, V=V, n_pad=n_pad, decay_is_log=log,
               use_l2norm=l2, scale=scale)
    pool = w.state_pool()
    p = problem(w, state=pool.copy())
    out = oracle.fwd(p)
    ref_out, finals = brute.fwd(w.qkv, w.decay, w.beta, pool, w.slot_idx, w.offsets,
                                nk=nk, nv=nv, K=K, V=V, decay_is_log=log, use_l2norm=l2,
                                scale=scale, eps=w.eps)
    np.testing.assert_allclose(out, ref_out, rtol=1e-10, atol=1e-12)
    touched = set()
    for (s, h), S in finals.items():
        touched.add((s, h))
        # the pool stores float32: the oracle's state is the float32 rounding of its
        # float64 state, which agrees with the matrix form to well under float32 ulp
        np.testing.assert_allclose(p.state[s, h], S, rtol=1e-6, atol=1e-7)
    for s in range(pool.shape[0]):
        for h in range(nv):
            if (s, h) not in touched:
                assert (p.state[s, h] == pool[s, h]).all()


def test_value_columns_split_into_independent_halves():
    """The value columns never mix: a V = 2K run equals, exactly, two V = K runs
    on the two halves of the value columns (v, state and output split alike)."""
    K = 16
    w = _small(15, [5, 2], nk=1, nv=2, K=K, V=2 * K, state_dtype="f32")
    pool = w.state_pool()
    p = problem(w, state=pool.copy())
    out = oracle.fwd(p)
    nv, qk = w.nv, 2 * w.nk * K
    for half in range(2):
        cols = slice(half * K, (half + 1) * K)
        v = w.qkv[:, qk:].reshape(-1, nv, 2 * K)[:, :, cols].reshape(-1, nv * K)
        wh = dataclasses.replace(w, V=K, qkv=np.concatenate([w.qkv[:, :qk], v], axis=1))
        ph = problem(wh, state=np.ascontiguousarray(pool[..., cols]))
        out_h = oracle.fwd(ph)
        assert (out.reshape(-1, nv, 2 * K)[:, :, cols] == out_h.reshape(-1, nv, K)).all()
        assert (p.state[..., cols] == ph.state).all()


def test_tiny_config_matches_bruteforce():
    w = W.tiny()
    pool = w.state_pool()
    ref_out, finals = brute.fwd(w.qkv, w.decay, w.beta, pool, w.slot_idx, w.offsets,
                                nk=w.nk, nv=w.nv, K=w.K, V=w.V)
    p = problem(w, state=pool.copy())
    out = oracle.fwd(p)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    for (slot, h), S in finals.items():
        np.testing.assert_allclose(p.state[slot, h], S, rtol=1e-6, atol=1e-7)
    untouched = [s for s in range(w.max_slots) if s not in w.live_slots()]
    for s in untouched:
        assert (p.state[s] == pool[s]).all()


def _golden():
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "exact_k4.json")
    with open(path) as f:
        return json.load(f)


def _golden_problem(g, use_l2norm):
    c = g["inputs"]
    pool = np.array(c["state"], dtype=np.float32)
    p = oracle.Problem(np.array(c["qkv"], np.float32), np.array(c["decay"], np.float32),
                       np.array(c["beta"], np.float32), pool, np.array(c["slot_idx"]),
                       np.array(c["offsets"]), nk=c["nk"], nv=c["nv"], K=c["K"], V=c["V"],
                       use_l2norm=use_l2norm, eps=0.0)
    return p


@pytest.mark.parametrize("use_l2norm", [True, False])
def test_matches_exact_rational_arithmetic(use_l2norm):
    """Exact rationals on a dyadic case: the float64 loops agree to ~1e-13."""
    g = _golden()
    c = g["inputs"]
    S0 = {s: c["state"][s] for s in range(len(c["state"]))}
    out_x, fin_x = exact.fwd_exact(c["qkv"], c["decay"], c["beta"], S0, c["slot_idx"],
                                   c["offsets"], nk=c["nk"], nv=c["nv"], K=c["K"], V=c["V"],
                                   use_l2norm=use_l2norm, eps=0)
    p = _golden_problem(g, use_l2norm)
    out = oracle.fwd(p)
    for (t, col), val in out_x.items():
        assert abs(out[t, col] - float(val)) <= 1e-13 * max(1.0, abs(float(val))), (t, col)
    for (slot, h), S in fin_x.items():
        want = np.array([[float(x) for x in row] for row in S])
        np.testing.assert_allclose(p.state[slot, h], want, rtol=2 ** -23, atol=1e-30)


def test_golden_fixture_exact_example():
    """tests/golden/exact_k4.json holds the exact rational outputs of the case."""
    g = _golden()
    p = _golden_problem(g, True)
    out = oracle.fwd(p)
    want = np.array([[float(Fraction(x)) for x in row] for row in g["out_exact"]])
    np.testing.assert_allclose(out, want, rtol=1e-13, atol=1e-15)
    for key, S in g["final_state_exact"].items():
        s, h = map(int, key.split(","))
        w = np.array([[float(Fraction(x)) for x in row] for row in S])
        np.testing.assert_allclose(p.state[s, h], w, rtol=2 ** -23, atol=1e-30)


# --------------------------------------------------------- closed forms ---

@pytest.mark.parametrize("work", ["f64", "f32"])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_beta0_decay1_leaves_state_unchanged(work, state_dtype):
    w = _small(3, [4, 2], nk=1, nv=2, K=16, state_dtype=state_dtype)
    w = dataclasses.replace(w, decay=np.ones_like(w.decay), beta=np.zeros_like(w.beta))
    pool = w.state_pool(w.live_slots())
    p = problem(w, state=pool.copy())
    oracle.fwd(p, work=work)
    assert (p.state == pool).all()


def test_decay1_beta1_unit_key_maps_key_to_value():
    """alpha=1, beta=1, |k^|=1: the updated state satisfies S^T k^ = v.  Read it
    out with q = k and scale = 1, so o = S^T k^ must equal v (and a readout taken
    before the update would not)."""
    w = _small(4, [1, 1, 1], nk=1, nv=2, K=16, state_dtype="f32")
    qkv = w.qkv.copy()
    K = w.K
    qkv[:, 0:K] = qkv[:, K:2 * K]  # q = k
    w = dataclasses.replace(w, qkv=qkv, decay=np.ones_like(w.decay), beta=np.ones_like(w.beta))
    p = problem(w, scale=1.0, eps=0.0)
    out = oracle.fwd(p)
    for b in range(w.batch):
        t = int(w.offsets[b])
        for h in range(w.nv):
            v = w.qkv[t, 2 * K + h * K: 2 * K + (h + 1) * K].astype(np.float64)
            np.testing.assert_allclose(out[t, h * K:(h + 1) * K], v, rtol=0, atol=1e-12)


def _qhat(qkv, t, hk, K, eps):
    q = qkv[t, hk * K:(hk + 1) * K].astype(np.float64)
    return q / np.sqrt(q @ q + eps)


def test_beta0_is_pure_decay_closed_form():
    """beta = 0: S_t = (prod alpha) S_0 and o_t = scale * (prod_{s<=t} alpha_s) S_0^T q^_t."""
    w = _small(5, [6, 3], nk=1, nv=2, K=16, state_dtype="f32")
    w = dataclasses.replace(w, beta=np.zeros_like(w.beta))
    pool = w.state_pool(w.live_slots())
    p = problem(w, state=pool.copy())
    out = oracle.fwd(p)
    scale = w.K ** -0.5
    for b in range(w.batch):
        slot = int(w.slot_idx[b])
        t0, t1 = int(w.offsets[b]), int(w.offsets[b + 1])
        for h in range(w.nv):
            S0 = pool[slot, h].astype(np.float64)
            prod = 1.0
            for t in range(t0, t1):
                prod *= float(w.decay[t, h])
                want = scale * prod * (S0.T @ _qhat(w.qkv, t, 0, w.K, w.eps))
                np.testing.assert_allclose(out[t, h * w.V:(h + 1) * w.V], want,
                                           rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(p.state[slot, h], prod * S0, rtol=2 ** -23, atol=0)


def test_zero_state_single_token_closed_form():
    """S_0 = 0, one token: o = scale * beta * (k^ . q^) * v (readout after the update)."""
    w = _small(6, [1, 1], nk=1, nv=2, K=16, state_dtype="f32")
    pool = np.zeros((w.max_slots, w.nv, w.K, w.V), np.float32)
    p = problem(w, state=pool)
    out = oracle.fwd(p)
    K = w.K
    for b in range(w.batch):
        t = int(w.offsets[b])
        q = _qhat(w.qkv, t, 0, K, w.eps)
        k = w.qkv[t, K:2 * K].astype(np.float64)
        k = k / np.sqrt(k @ k + w.eps)
        for h in range(w.nv):
            v = w.qkv[t, 2 * K + h * K: 2 * K + (h + 1) * K].astype(np.float64)
            want = K ** -0.5 * float(w.beta[t, h]) * (k @ q) * v
            np.testing.assert_allclose(out[t, h * K:(h + 1) * K], want, rtol=1e-12, atol=1e-15)


def test_scale_argument_multiplies_output():
    w = _small(7, [3], nk=1, nv=2, K=16)
    o1 = oracle.fwd(problem(w, scale=0.0))
    o2 = oracle.fwd(problem(w, scale=0.5))
    np.testing.assert_allclose(o2, o1 * (0.5 / w.K ** -0.5), rtol=1e-13, atol=0)


def test_l2norm_is_scale_invariant_in_q_and_k():
    w = _small(8, [5, 2], nk=2, nv=4, K=16)
    qkv = w.qkv.copy()
    nkK = w.nk * w.K
    qkv[:, :nkK] *= np.float32(4.0)        # q scaled by an exact power of two
    qkv[:, nkK:2 * nkK] *= np.float32(0.25)  # k likewise
    o1 = oracle.fwd(problem(w, eps=0.0))
    o2 = oracle.fwd(problem(dataclasses.replace(w, qkv=qkv), eps=0.0))
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-14)


def test_log_decay_equals_exp_decay():
    w = _small(9, [4, 3], nk=1, nv=2, K=16, decay_is_log=True)
    ref, _ = brute.fwd(w.qkv, w.decay, w.beta, w.state_pool(w.live_slots()), w.slot_idx,
                       w.offsets, nk=1, nv=2, K=16, V=16, decay_is_log=True)
    out = oracle.fwd(problem(w))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------ invariants ---

def test_padding_rows_zero_output_and_untouched_pool():
    w = _small(10, [3, 4, 2], nk=1, nv=2, K=16, n_pad=1)
    pool = w.state_pool()
    p = problem(w, state=pool.copy())
    out = oracle.fwd(p)
    for b in range(w.batch):
        if w.slot_idx[b] < 0:
            t0, t1 = int(w.offsets[b]), int(w.offsets[b + 1])
            assert (out[t0:t1] == 0).all()
    touched = set(w.live_slots())
    for s in range(w.max_slots):
        if s not in touched:
            assert (p.state[s] == pool[s]).all()


def test_empty_rows_leave_state_alone():
    w = _small(12, [0, 3, 0], nk=1, nv=2, K=16)
    pool = w.state_pool()
    p = problem(w, state=pool.copy())
    oracle.fwd(p)
    for b in (0, 2):
        s = int(w.slot_idx[b])
        assert (p.state[s] == pool[s]).all()


def test_rows_are_independent_and_order_free():
    w = _small(13, [3, 5, 1, 4], nk=2, nv=4, K=16)
    pool = w.state_pool()
    p = problem(w, state=pool.copy())
    out = oracle.fwd(p)
    for b in [2, 0, 3, 1]:
        sub = sub_workload(w, [b])
        ps = problem(sub, state=pool.copy())
        o = oracle.fwd(ps)
        t0, t1 = int(w.offsets[b]), int(w.offsets[b + 1])
        assert (o == out[t0:t1]).all()
        s = int(w.slot_idx[b])
        assert (ps.state[s] == p.state[s]).all()


def test_gqa_matches_duplicated_key_heads():
    """nk key heads shared by r value heads == nk*r key heads holding copies."""
    w = _small(14, [4, 3], nk=2, nv=4, K=16)
    K, nk, nv = w.K, w.nk, w.nv
    r = nv // nk
    q = w.qkv[:, :nk * K].reshape(-1, nk, K)
    k = w.qkv[:, nk * K:2 * nk * K].reshape(-1, nk, K)
    v = w.qkv[:, 2 * nk * K:]
    q2 = np.repeat(q, r, axis=1).reshape(len(q), -1)
    k2 = np.repeat(k, r, axis=1).reshape(len(k), -1)
    w2 = dataclasses.replace(w, nk=nv, qkv=np.concatenate([q2, k2, v], axis=1))
    pool = w.state_pool()
    p1 = problem(w, state=pool.copy())
    p2 = problem(w2, state=pool.copy())
    assert (oracle.fwd(p1) == oracle.fwd(p2)).all()
    assert (p1.state == p2.state).all()


def test_chaining_split_rows_bitwise_in_float32():
    """float32 pool and float32 work: running a row in two calls equals one call."""
    w = _small(15, [7, 5], nk=1, nv=2, K=16, state_dtype="f32")
    pool = w.state_pool()
    p = problem(w, state=pool.copy())
    out = oracle.fwd(p, work="f32")
    split = [3, 2]
    first = dataclasses.replace(
        w, offsets=np.array([0, 3, 3 + 2], np.int32),
        qkv=np.concatenate([w.qkv[0:3], w.qkv[7:9]]),
        decay=np.concatenate([w.decay[0:3], w.decay[7:9]]),
        beta=np.concatenate([w.beta[0:3], w.beta[7:9]]))
    second = dataclasses.replace(
        w, offsets=np.array([0, 4, 4 + 3], np.int32),
        qkv=np.concatenate([w.qkv[3:7], w.qkv[9:12]]),
        decay=np.concatenate([w.decay[3:7], w.decay[9:12]]),
        beta=np.concatenate([w.beta[3:7], w.beta[9:12]]))
    st = pool.copy()
    o1 = oracle.fwd(problem(first, state=st), work="f32")
    o2 = oracle.fwd(problem(second, state=st), work="f32")
    assert (st == p.state).all()
    assert (np.concatenate([o1[0:3], o2[0:4], o1[3:5], o2[4:7]]) == out).all()
    del split


def test_invalid_arguments_rejected():
    w = _small(16, [2], nk=1, nv=2, K=16)
    pool = w.state_pool()
    with pytest.raises(ValueError):  # slot beyond the pool
        oracle.fwd(problem(dataclasses.replace(w, slot_idx=np.array([w.max_slots], np.int32)),
                           state=pool.copy()))
    with pytest.raises(ValueError):  # row end beyond total tokens
        oracle.fwd(problem(dataclasses.replace(w, offsets=np.array([0, 3], np.int32)),
                           state=pool.copy()))
    with pytest.raises(ValueError):  # nv not a multiple of nk (qkv shaped for nk=3)
        K = w.K
        qkv = np.zeros((w.total_tokens, 2 * 3 * K + w.nv * K), np.float32)
        oracle.fwd(problem(dataclasses.replace(w, qkv=qkv), state=pool.copy(), nk=3))


# ------------------------------------------------- per-element beta ---

def test_beta_per_value_columns_equal_headwise_runs():
    """beta [T, HV, V] ("core.ssm.ops.gdp.fused_recurrent" Parameters): the
    columns of S evolve independently (each sees only its own a_j, u_j), so
    column j of a run with per-element beta equals, exactly, column j of a run
    whose head-wise beta is that column's value."""
    levels = np.array([0.0, 0.25, 0.5, 1.0], np.float32)
    w = _small(40, [4, 3], nk=1, nv=2, K=16, state_dtype="f32")
    T, nv, V = w.total_tokens, w.nv, w.V
    rng = np.random.default_rng(41)
    pick = rng.integers(0, len(levels), size=(nv, V))       # one level per (head, column)
    beta_pv = np.broadcast_to(levels[pick], (T, nv, V)).astype(np.float32).copy()
    pool = w.state_pool()
    pp = problem(dataclasses.replace(w, beta=beta_pv), state=pool.copy())
    out_pv = oracle.fwd(pp)
    for li, lv in enumerate(levels):
        ph = problem(dataclasses.replace(w, beta=np.full((T, nv), lv, np.float32)), state=pool.copy())
        out_h = oracle.fwd(ph)
        for h in range(nv):
            cols = np.nonzero(pick[h] == li)[0]
            if cols.size == 0:
                continue
            assert (out_pv[:, h * V + cols] == out_h[:, h * V + cols]).all()
            for s in w.slot_idx:
                assert (pp.state[s, h][:, cols] == ph.state[s, h][:, cols]).all()


def test_beta_per_value_zero_column_only_decays():
    """beta_j = 0 makes u_j = 0: column j of S is only decayed, token by token."""
    w = _small(42, [3], nk=1, nv=1, K=16, state_dtype="f32")
    T, V = w.total_tokens, w.V
    beta = np.full((T, 1, V), 0.7, np.float32)
    beta[:, 0, 5] = 0.0
    pool = w.state_pool()
    p = problem(dataclasses.replace(w, beta=beta), state=pool.copy())
    oracle.fwd(p)
    s = int(w.slot_idx[0])
    decay = np.prod(w.decay[:, 0].astype(np.float64))
    np.testing.assert_allclose(p.state[s, 0][:, 5], decay * pool[s, 0][:, 5].astype(np.float64),
                               rtol=1e-6)
    assert not np.allclose(p.state[s, 0][:, 4], decay * pool[s, 0][:, 4])


# --------------------------------------------- dense initial / final state ---

def _dense_inputs(w):
    return dict(nk=w.nk, nv=w.nv, K=w.K, V=w.V, state_dtype=w.state_dtype, decay_is_log=w.decay_is_log,
                use_l2norm=w.use_l2norm, scale=w.scale, eps=w.eps)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_dense_state_equals_pool_at_the_rows_slots(state_dtype):
    """initial_state / output_final_state ("core.ssm.ops.gdp.fused_recurrent"
    Parameters) is the slot-indexed pass with the rows' states gathered densely:
    same output, final[n] = the pool slot of row n after the pass, and an empty
    row returns its initial state."""
    w = _small(50, [4, 0, 7], nk=1, nv=2, K=16, state_dtype=state_dtype)
    pool = w.state_pool()
    pp = problem(w, state=pool.copy())
    out_pool = oracle.fwd(pp)
    init = pool[w.slot_idx].copy()
    out_d, final = oracle.fwd_dense(w.qkv, w.decay, w.beta, w.offsets, init, **_dense_inputs(w))
    assert (out_d == out_pool).all()
    assert (final == pp.state[w.slot_idx]).all()
    assert (final[1] == init[1]).all()


def test_dense_state_without_initial_state_starts_from_zero():
    """initial_state None means zeros: one token from S_0 = 0 gives
    o = scale * beta * (k^ . q^) * v (readout of the updated state) and the
    final state beta k^ v^T."""
    w = _small(51, [1], nk=1, nv=1, K=16, state_dtype="f32")
    out, final = oracle.fwd_dense(w.qkv, w.decay, w.beta, w.offsets, None, **_dense_inputs(w))
    K = w.K
    q = w.qkv[0, :K].astype(np.float64)
    k = w.qkv[0, K:2 * K].astype(np.float64)
    v = w.qkv[0, 2 * K:].astype(np.float64)
    qh, kh = q / np.sqrt(q @ q + w.eps), k / np.sqrt(k @ k + w.eps)
    b = float(w.beta[0, 0])
    np.testing.assert_allclose(out[0], K ** -0.5 * b * (kh @ qh) * v, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(final[0, 0], (b * np.outer(kh, v)).astype(np.float32), rtol=1e-6)


# ---------------------------------------------------------- verify / fold ---

def _ring(w, nk, ring_len, rows, bf16=False):
    stride = oracle.ring_record_elements(w.K, w.V, w.nv // nk)
    stride = (stride + 7) // 8 * 8
    if bf16:  # 0x7FC0 is a bfloat16 NaN
        return np.full((rows, nk, ring_len, stride), 0x7FC0, np.uint16)
    return np.full((rows, nk, ring_len, stride), np.nan, np.float32)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_verify_output_equals_forward_and_pool_untouched(state_dtype):
    w = _small(20, [3, 5, 2, 9], nk=2, nv=4, K=16, n_pad=1, state_dtype=state_dtype)
    ring_len = 8
    rsi = np.array([3, 1, 0, 2], np.int32)
    pool = w.state_pool()
    pf = problem(w, state=pool.copy())
    out_f = oracle.fwd(pf)
    pv = problem(w, state=pool.copy())
    ring = _ring(w, w.nk, ring_len, 4)
    out_v = oracle.verify_ring(pv, ring, rsi, ring_len)
    assert (out_v == out_f).all()
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        if s < 0:
            continue
        L = int(w.row_lengths[b])
        if L <= ring_len:
            assert (pv.state[s] == pool[s]).all(), "verify must not write the pool"
        else:
            # a row longer than RING_LEN commits like the forward pass and records nothing
            assert (pv.state[s] == pf.state[s]).all()
            assert np.isnan(ring[rsi[b]]).all()


def test_verify_records_hold_normalised_key_alpha_and_correction():
    w = _small(21, [2], nk=1, nv=2, K=16, state_dtype="f32")
    ring_len = 4
    pool = w.state_pool()
    ring = _ring(w, 1, ring_len, 1)
    oracle.verify_ring(problem(w, state=pool.copy()), ring, np.array([0], np.int32), ring_len)
    K = V = w.K
    t = 0
    k = w.qkv[t, K:2 * K].astype(np.float64)
    kh = k / np.sqrt(k @ k + w.eps)
    rec = ring[0, 0, 0]
    np.testing.assert_allclose(rec[:K], kh, rtol=2 ** -23)
    slot = int(w.slot_idx[0])
    for h in range(2):
        alpha = float(w.decay[t, h])
        assert rec[K + h] == np.float32(alpha)
        S = alpha * pool[slot, h].astype(np.float64)
        v = w.qkv[t, 2 * K + h * V: 2 * K + (h + 1) * V].astype(np.float64)
        u = float(w.beta[t, h]) * (v - S.T @ kh)
        np.testing.assert_allclose(rec[K + 8 + h * V: K + 8 + (h + 1) * V], u, rtol=1e-6,
                                   atol=1e-7)
    assert np.isnan(ring[0, 0, 2:]).all()  # only two tokens recorded


def test_row_of_exactly_ring_len_records():
    w = _small(22, [4, 5], nk=1, nv=2, K=16)
    ring = _ring(w, 1, 4, 2)
    pool = w.state_pool()
    pv = problem(w, state=pool.copy())
    oracle.verify_ring(pv, ring, np.array([0, 1], np.int32), 4)
    K, r = w.K, w.nv
    fields = np.r_[0:K, K:K + r, K + 8:K + 8 + r * w.V]  # k^, alpha_j, u_j (not the pad)
    assert not np.isnan(ring[0][..., fields]).any()     # L == RING_LEN records
    assert np.isnan(ring[1]).all()              # L == RING_LEN + 1 commits instead
    assert (pv.state[w.slot_idx[0]] == pool[w.slot_idx[0]]).all()
    assert not (pv.state[w.slot_idx[1]] == pool[w.slot_idx[1]]).all()


def test_bf16_ring_records_are_the_float32_records_rounded():
    """A bfloat16 ring ("gated_delta_recurrence_verify_ring_gpu" Parameters:
    ring_dtype) holds each record value rounded to nearest-even once: from the
    float64 oracle's value, the bits equal rounding that value directly."""
    w = _small(23, [3, 2], nk=2, nv=4, K=16, state_dtype="bf16", n_pad=1)
    rsi = np.array([1, 0, 2], np.int32)
    pool = w.state_pool()
    r32 = _ring(w, w.nk, 4, 3)
    r16 = _ring(w, w.nk, 4, 3, bf16=True)
    # the float64 values behind the float32 ring: rerun the verify in float64 and
    # compare bfloat16 bits with the float32 ring rounded from float64 where the
    # float32 rounding cannot move a bfloat16 decision
    out32 = oracle.verify_ring(problem(w, state=pool.copy()), r32, rsi, 4)
    out16 = oracle.verify_ring(problem(w, state=pool.copy()), r16, rsi, 4)
    assert (out32 == out16).all(), "the ring dtype does not change the output"
    written = ~np.isnan(r32)
    assert (written == (r16 != 0x7FC0)).all(), "same fields written"
    wide = oracle.bf16_to_f64(r16[written])
    ref = r32[written].astype(np.float64)
    # bfloat16 keeps 8 significant bits: within half a bfloat16 ulp of the value
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
    assert (np.abs(wide - ref) <= ulp / 2 * (1 + 2 ** -16)).all()
    # and on bfloat16-representable values the rounding is the identity
    exact = oracle.round_bf16(wide)
    assert (exact == r16[written]).all()


def test_bf16_ring_fold_equals_float32_ring_fold_on_representable_records():
    """Folding records whose values are bfloat16-representable gives the same
    state from a float32 and from a bfloat16 ring: the fold only widens."""
    w = _small(24, [1, 1, 1], nk=1, nv=2, K=16, state_dtype="f32")
    stride = (oracle.ring_record_elements(16, 16, 2) + 7) // 8 * 8
    rng = np.random.default_rng(25)
    vals = rng.standard_normal((3, 1, 4, stride)) * 0.3
    vals[..., 16:18] = rng.uniform(0.8, 1.0, (3, 1, 4, 2))
    r16 = oracle.round_bf16(vals)
    r32 = oracle.bf16_to_f64(r16).astype(np.float32)
    counts = np.array([3, 0, 4], np.int32)
    rsi = np.array([2, 0, 1], np.int32)
    pool = w.state_pool()
    p32, p16 = problem(w, state=pool.copy()), problem(w, state=pool.copy())
    oracle.fold(p32, r32, rsi, counts, 4)
    oracle.fold(p16, r16, rsi, counts, 4)
    assert (p32.state == p16.state).all()
    assert not (p32.state == pool).all()


def test_bf16_ring_fold_tracks_the_forward_pass():
    """verify + fold(c) with a bfloat16 ring stays within the records' rounding
    of the forward pass over the first c tokens (not bit-exact: the pages keep
    bit-exactness for float32 rings only)."""
    w = _small(26, [5, 4], nk=1, nv=2, K=16, state_dtype="f32")
    counts = np.array([3, 4], np.int32)
    rsi = np.array([1, 0], np.int32)
    pool = w.state_pool()
    pv = problem(w, state=pool.copy())
    ring = _ring(w, 1, 8, 2, bf16=True)
    oracle.verify_ring(pv, ring, rsi, 8)
    oracle.fold(pv, ring, rsi, counts, 8)
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        c = int(counts[b])
        sub = dataclasses.replace(sub_workload(w, [b]), offsets=np.array([0, c], np.int32))
        sub = dataclasses.replace(sub, qkv=sub.qkv[:c], decay=sub.decay[:c], beta=sub.beta[:c])
        pf = problem(sub, state=pool.copy())
        oracle.fwd(pf)
        d = np.abs(pv.state[s].astype(np.float64) - pf.state[s])
        assert d.max() < 2e-2 and d.max() > 0


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_fold_equals_forward_over_accepted_prefix_bitwise_float32(state_dtype):
    """With float32 work and a float32 ring, verify + fold(c) == forward over the
    first c tokens, bit for bit ("gated_delta_recurrence_verify_ring_gpu",
    ring_dtype: bit-exact only for float32)."""
    lengths = [5, 5, 3, 5, 5, 12]
    w = _small(23, lengths, nk=2, nv=4, K=16, state_dtype=state_dtype, n_pad=1)
    ring_len = 8
    counts = np.array([0, 1, 3, 5, 4, 12], np.int32)
    rsi = np.arange(w.batch, dtype=np.int32)[::-1].copy()
    pool = w.state_pool()
    pv = problem(w, state=pool.copy())
    ring = _ring(w, w.nk, ring_len, w.batch)
    oracle.verify_ring(pv, ring, rsi, ring_len, work="f32")
    oracle.fold(pv, ring, rsi, counts, ring_len, work="f32")
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        if s < 0:
            continue
        L = int(w.row_lengths[b])
        c = int(counts[b])
        if L > ring_len:
            # committed by verify; the fold skips count > RING_LEN
            pf = problem(sub_workload(w, [b]), state=pool.copy())
            oracle.fwd(pf, work="f32")
            assert (pv.state[s] == pf.state[s]).all()
            continue
        pref = sub_workload(w, [b])
        pref = dataclasses.replace(pref, offsets=np.array([0, c], np.int32),
                                   qkv=pref.qkv[:c], decay=pref.decay[:c], beta=pref.beta[:c])
        pf = problem(pref, state=pool.copy())
        oracle.fwd(pf, work="f32")
        assert (pv.state[s] == pf.state[s]).all(), (b, c)


@pytest.mark.parametrize("seed", range(8))
def test_random_verify_fold_equals_prefix_forward(seed):
    """The same contract over random small shapes: GQA groups of 1 or 2, K from
    4 to 16, either decay form, either pool type, ragged rows around RING_LEN,
    accepted counts from 0 to the row's length, rows in shuffled ring rows."""
    rng = np.random.default_rng(3000 + seed)
    nk = int(rng.choice([1, 2]))
    nv = nk * int(rng.choice([1, 2]))
    K = int(rng.choice([4, 8, 16]))
    ring_len = int(rng.choice([2, 4, 8]))
    lengths = [int(x) for x in rng.integers(0, ring_len + 3, size=int(rng.integers(2, 7)))]
    state_dtype = str(rng.choice(["f32", "bf16"]))
    log = bool(rng.integers(0, 2))
    w = _small(4000 + seed, lengths, nk=nk, nv=nv, K=K, state_dtype=state_dtype,
               n_pad=int(rng.integers(0, 2)), decay_is_log=log)
    # an accepted count is at most the row's length; a row longer than RING_LEN
    # is committed by the verify pass and recorded nothing, so its count is past
    # RING_LEN (the fold must skip it)
    counts = np.array([L if L > ring_len else int(rng.integers(0, L + 1)) for L in lengths],
                      np.int32)
    rsi = rng.permutation(w.batch).astype(np.int32)
    pool = w.state_pool()
    pv = problem(w, state=pool.copy())
    ring = _ring(w, w.nk, ring_len, w.batch)
    oracle.verify_ring(pv, ring, rsi, ring_len, work="f32")
    oracle.fold(pv, ring, rsi, counts, ring_len, work="f32")
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        if s < 0:
            continue
        L, c = int(w.row_lengths[b]), int(counts[b])
        # rows longer than RING_LEN commit in the verify pass; the fold skips
        # counts of zero or past RING_LEN; otherwise the first c tokens count
        n = L if L > ring_len else (c if 0 < c <= ring_len else 0)
        if n == 0:
            assert (pv.state[s] == pool[s]).all(), (b, L, c)
            continue
        pref = sub_workload(w, [b])
        pref = dataclasses.replace(pref, offsets=np.array([0, n], np.int32),
                                   qkv=pref.qkv[:n], decay=pref.decay[:n], beta=pref.beta[:n])
        pf = problem(pref, state=pool.copy())
        oracle.fwd(pf, work="f32")
        assert (pv.state[s] == pf.state[s]).all(), (b, L, c)


def test_fold_float64_close_to_prefix_forward():
    w = _small(24, [5, 5], nk=1, nv=2, K=16, state_dtype="f32")
    counts = np.array([2, 5], np.int32)
    pool = w.state_pool()
    pv = problem(w, state=pool.copy())
    ring = _ring(w, 1, 8, 2)
    rsi = np.array([0, 1], np.int32)
    oracle.verify_ring(pv, ring, rsi, 8)
    oracle.fold(pv, ring, rsi, counts, 8)
    for b in range(2):
        c = int(counts[b])
        pref = sub_workload(w, [b])
        pref = dataclasses.replace(pref, offsets=np.array([0, c], np.int32),
                                   qkv=pref.qkv[:c], decay=pref.decay[:c], beta=pref.beta[:c])
        pf = problem(pref, state=pool.copy())
        oracle.fwd(pf)
        s = int(w.slot_idx[b])
        np.testing.assert_allclose(pv.state[s], pf.state[s], rtol=1e-6, atol=1e-7)


def test_fold_skips_zero_too_many_and_padding():
    w = _small(25, [3, 3, 3], nk=1, nv=2, K=16, n_pad=0)
    w = dataclasses.replace(w, slot_idx=np.array([w.slot_idx[0], w.slot_idx[1], -1], np.int32))
    pool = w.state_pool()
    pv = problem(w, state=pool.copy())
    stride = oracle.ring_record_elements(16, 16, 2)
    ring = np.random.default_rng(0).standard_normal((3, 1, 4, stride)).astype(np.float32)
    oracle.fold(pv, ring, np.array([0, 1, 2], np.int32), np.array([0, 5, 2], np.int32), 4)
    assert (pv.state == pool).all()


# ------------------------------------------------- snapshots / rollback ---

@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_snapshots_equal_prefix_forward_and_rollback(state_dtype):
    """intermediate_states[slot, i] == state after the first (i+1)*spt steps;
    rollback(a) restores exactly that ("core.ssm.ops.gdp.fused_recurrent",
    intermediate_states / steps_per_token)."""
    spt, drafts = 2, 4
    w = _small(30, [8, 8, 7, 8], nk=2, nv=4, K=16, state_dtype=state_dtype, n_pad=1,
               decay_is_log=True)
    pool = w.state_pool()
    dt = pool.dtype
    inter = np.full((w.max_slots, drafts, w.nv, w.K, w.V),
                    0xFFFF if dt == np.uint16 else np.nan, dtype=dt)
    ps = problem(w, state=pool.copy())
    out_s = oracle.fwd_snapshots(ps, inter, spt)
    pf = problem(w, state=pool.copy())
    assert (oracle.fwd(pf) == out_s).all()
    assert (pf.state == ps.state).all()
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        if s < 0:
            continue
        L = int(w.row_lengths[b])
        for i in range(drafts):
            n = (i + 1) * spt
            if n > L:  # partial trailing draft: not snapshotted
                if dt == np.uint16:
                    assert (inter[s, i] == 0xFFFF).all()
                else:
                    assert np.isnan(inter[s, i]).all()
                continue
            pref = sub_workload(w, [b])
            pref = dataclasses.replace(pref, offsets=np.array([0, n], np.int32),
                                       qkv=pref.qkv[:n], decay=pref.decay[:n], beta=pref.beta[:n])
            pp = problem(pref, state=pool.copy())
            oracle.fwd(pp)
            assert (inter[s, i] == pp.state[s]).all(), (b, i)
        if L == drafts * spt:
            assert (inter[s, drafts - 1] == ps.state[s]).all()
    # padding wrote nothing anywhere
    live = set(w.live_slots())
    for s in range(w.max_slots):
        if s not in live:
            if dt == np.uint16:
                assert (inter[s] == 0xFFFF).all()
            else:
                assert np.isnan(inter[s]).all()
    # rollback: rows with a complete snapshot at the accepted index
    acc = np.array([1, 0, 2, 3], np.int32)
    acc[w.slot_idx < 0] = -1
    acc[2] = 2 if w.row_lengths[2] >= 6 else 0
    pr = problem(w, state=ps.state.copy())
    oracle.rollback(pr, inter, acc)
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        if s < 0:
            continue
        assert (pr.state[s] == inter[s, acc[b]]).all()


@pytest.mark.parametrize("seed", range(8))
def test_random_snapshots_equal_prefix_forward(seed):
    """The snapshot contract over random small shapes: steps per token 1 to 3,
    2 to 4 snapshot slots, rows that end mid-draft or hold fewer drafts than
    the slots, either pool type and decay form."""
    rng = np.random.default_rng(5000 + seed)
    nk = int(rng.choice([1, 2]))
    nv = nk * int(rng.choice([1, 2]))
    K = int(rng.choice([4, 8]))
    spt = int(rng.integers(1, 4))
    drafts = int(rng.integers(2, 5))
    lengths = [int(x) for x in rng.integers(0, drafts * spt + 1, size=int(rng.integers(2, 6)))]
    state_dtype = str(rng.choice(["f32", "bf16"]))
    w = _small(6000 + seed, lengths, nk=nk, nv=nv, K=K, state_dtype=state_dtype,
               n_pad=int(rng.integers(0, 2)), decay_is_log=bool(rng.integers(0, 2)))
    pool = w.state_pool()
    dt = pool.dtype
    blank = 0xFFFF if dt == np.uint16 else np.nan
    inter = np.full((w.max_slots, drafts, w.nv, w.K, w.V), blank, dtype=dt)
    ps = problem(w, state=pool.copy())
    oracle.fwd_snapshots(ps, inter, spt)
    for b in range(w.batch):
        s = int(w.slot_idx[b])
        if s < 0:
            continue
        L = int(w.row_lengths[b])
        for i in range(drafts):
            n = (i + 1) * spt
            if n > L:  # not reached: nothing written
                if dt == np.uint16:
                    assert (inter[s, i] == blank).all()
                else:
                    assert np.isnan(inter[s, i]).all()
                continue
            pref = sub_workload(w, [b])
            pref = dataclasses.replace(pref, offsets=np.array([0, n], np.int32),
                                       qkv=pref.qkv[:n], decay=pref.decay[:n], beta=pref.beta[:n])
            pp = problem(pref, state=pool.copy())
            oracle.fwd(pp)
            assert (inter[s, i] == pp.state[s]).all(), (b, i)


def test_gdp_config_folding_structure():
    """Config-5 input structure: decay only on the first Householder copy."""
    w = W.gdp_snapshots(batch=2, nk=1, nv=2, K=16, max_slots=4)
    M = w.steps_per_token
    step = np.arange(w.total_tokens) % (w.meta["drafts"] * M)
    assert (w.decay[step % M != 0] == 0).all()
    assert (w.decay[step % M == 0] < 0).all()
