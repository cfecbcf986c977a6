"""Matrix-form brute force for tiny cases -- TEST INFRASTRUCTURE ONLY.

An independent numpy statement of the gated delta rule used to pin the C loop
oracle.  Instead of the four elementwise steps it applies the closed matrix
update per token,

    S_t = alpha_t * (I - beta_t k^_t k^_t^T) S_{t-1} + beta_t k^_t v_t^T
    o_t = scale * S_t^T q^_t

("core.ssm.ops.gdp.fused_recurrent": fused recurrent gated delta rule step;
"gated_delta_recurrence_fwd_gpu": L2-normalised q/k and K^-0.5 query scale),
built with np.eye / np.outer / @ in float64, one (row, head) at a time.
"""
from __future__ import annotations

import numpy as np


def _state_f64(state):
    if state.dtype == np.uint16:
        return (state.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return state.astype(np.float64)


def fwd(qkv, decay, beta, state, slot_idx, offsets, *, nk, nv, K, V,
        decay_is_log=False, use_l2norm=True, scale=0.0, eps=1e-6):
    """Returns (out [T, nv*V], final float64 states {(slot, h): S}) without
    touching ``state``; float64 throughout, no storage rounding."""
    T = qkv.shape[0]
    r = nv // nk
    scale = scale if scale > 0 else K ** -0.5
    S_all = _state_f64(state)
    out = np.zeros((T, nv * V))
    finals = {}
    for b in range(len(slot_idx)):
        t0, t1 = int(offsets[b]), int(offsets[b + 1])
        slot = int(slot_idx[b])
        if slot < 0:
            continue
        for h in range(nv):
            hk = h // r
            S = S_all[slot, h].copy()
            for t in range(t0, t1):
                q = qkv[t, hk * K:(hk + 1) * K].astype(np.float64)
                k = qkv[t, nk * K + hk * K: nk * K + (hk + 1) * K].astype(np.float64)
                v = qkv[t, 2 * nk * K + h * V: 2 * nk * K + (h + 1) * V].astype(np.float64)
                if use_l2norm:
                    q = q / np.sqrt(q @ q + eps)
                    k = k / np.sqrt(k @ k + eps)
                a = float(decay[t, h])
                a = np.exp(a) if decay_is_log else a
                bt = float(beta[t, h])
                S = a * (np.eye(K) - bt * np.outer(k, k)) @ S + bt * np.outer(k, v)
                out[t, h * V:(h + 1) * V] = scale * (S.T @ q)
            finals[(slot, h)] = S
    return out, finals
