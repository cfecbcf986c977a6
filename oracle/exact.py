"""Exact rational restatement of the recurrence for tiny cases -- TEST INFRASTRUCTURE ONLY.

Uses fractions.Fraction throughout, so the result carries no rounding at all.
Inputs must be exactly representable (dyadic values stored in float32), and
when L2 normalisation is on the squared norms plus eps must be perfect
squares of rationals (e.g. k = (1, 2, 2, 4) has norm 5 with eps = 0).

Per token, for one (sequence, value head) -- "gated_delta_recurrence_fwd_gpu"
summary and "core.ssm.ops.gdp.fused_recurrent" parameters:
    S <- alpha S ;  u = beta (v - S^T k^) ;  S <- S + k^ u^T ;  o = scale S^T q^
"""
from __future__ import annotations

from fractions import Fraction
from math import isqrt


def _sqrt_exact(x: Fraction) -> Fraction:
    n, d = x.numerator, x.denominator
    rn, rd = isqrt(n), isqrt(d)
    if rn * rn != n or rd * rd != d:
        raise ValueError(f"{x} is not the square of a rational")
    return Fraction(rn, rd)


def fwd_exact(qkv, decay, beta, S0, slot_idx, offsets, *, nk, nv, K, V,
              use_l2norm=False, scale=None, eps=0):
    """qkv/decay/beta: nested lists of numbers; S0: dict slot -> [nv][K][V].
    Returns (out as {(t, h*V+j): Fraction}, final {(slot, h): [[Fraction]]})."""
    r = nv // nk
    if scale is None:
        scale = 1 / _sqrt_exact(Fraction(K))
    scale = Fraction(scale)
    eps = Fraction(eps)
    out, finals = {}, {}
    for b in range(len(slot_idx)):
        slot = slot_idx[b]
        t0, t1 = offsets[b], offsets[b + 1]
        for h in range(nv):
            if slot < 0:
                for t in range(t0, t1):
                    for j in range(V):
                        out[(t, h * V + j)] = Fraction(0)
                continue
            hk = h // r
            S = [[Fraction(x) for x in row] for row in S0[slot][h]]
            for t in range(t0, t1):
                q = [Fraction(x) for x in qkv[t][hk * K:(hk + 1) * K]]
                k = [Fraction(x) for x in qkv[t][nk * K + hk * K: nk * K + (hk + 1) * K]]
                v = [Fraction(x) for x in qkv[t][2 * nk * K + h * V: 2 * nk * K + (h + 1) * V]]
                if use_l2norm:
                    nq = _sqrt_exact(sum(x * x for x in q) + eps)
                    nkk = _sqrt_exact(sum(x * x for x in k) + eps)
                    q = [x / nq for x in q]
                    k = [x / nkk for x in k]
                a = Fraction(decay[t][h])
                bt = Fraction(beta[t][h])
                S = [[a * S[i][j] for j in range(V)] for i in range(K)]
                u = [bt * (v[j] - sum(S[i][j] * k[i] for i in range(K))) for j in range(V)]
                S = [[S[i][j] + k[i] * u[j] for j in range(V)] for i in range(K)]
                for j in range(V):
                    out[(t, h * V + j)] = scale * sum(S[i][j] * q[i] for i in range(K))
            finals[(slot, h)] = S
    return out, finals
