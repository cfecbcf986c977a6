"""Seeded synthetic inputs for the gated delta rule path.

This module only draws random numbers and lays them out; it contains none of
the recurrence's arithmetic, so both the CPU oracle and the CUDA library can
consume what it produces.  All arrays are host numpy arrays in the layouts of
"gated_delta_recurrence_fwd_gpu" (Args):

  qkv      [T, 2*nk*K + nv*V] float32: Q | K | V channel ranges, heads contiguous
  decay    [T, nv] float32: multiplicative decay alpha, or log decay g
  beta     [T, nv] float32, or [T, nv, V] per value element
           ("core.ssm.ops.gdp.fused_recurrent", beta [B, T, HV] or [B, T, HV, V])
  state    [slots, nv, K, V]: float32, or uint16 holding bfloat16 bits
  slot_idx [batch] int32, -1 = padding request
  offsets  [batch+1] int32, row b spans [offsets[b], offsets[b+1])

Pool contents are drawn per slot from their own stream (seed, slot), so a test
can materialise only the slots it reads.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits (round to nearest even) via torch's CPU cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


@dataclass
class Workload:
    name: str
    nk: int
    nv: int
    K: int
    V: int
    qkv: np.ndarray
    decay: np.ndarray
    beta: np.ndarray
    slot_idx: np.ndarray
    offsets: np.ndarray
    max_slots: int
    state_dtype: str                       # "bf16" or "f32"
    state_seed: int
    state_std: float
    decay_is_log: bool = False
    use_l2norm: bool = True
    scale: float = 0.0                     # <= 0: K^-0.5
    eps: float = 1e-6
    # speculative decoding extras
    ring_len: int = 0
    ring_rows: int = 0
    ring_slot_idx: Optional[np.ndarray] = None
    counts: Optional[np.ndarray] = None
    steps_per_token: int = 1
    n_inter: int = 0
    accepted: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.slot_idx.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(self.qkv.shape[0])

    @property
    def row_lengths(self) -> np.ndarray:
        return np.diff(self.offsets.astype(np.int64))

    @property
    def live_head_tokens(self) -> int:
        live = self.slot_idx >= 0
        return int(self.row_lengths[live].sum()) * self.nv

    def state_slot(self, slot: int) -> np.ndarray:
        """Initial contents of one pool slot, [nv, K, V]."""
        rng = np.random.default_rng([self.state_seed, 7919, int(slot)])
        x = rng.standard_normal((self.nv, self.K, self.V), dtype=np.float32) * np.float32(self.state_std)
        return _bf16_bits(x) if self.state_dtype == "bf16" else x

    def state_pool(self, slots=None) -> np.ndarray:
        """The initial pool [max_slots, nv, K, V]; only ``slots`` are drawn
        (others zero) when given."""
        dt = np.uint16 if self.state_dtype == "bf16" else np.float32
        pool = np.zeros((self.max_slots, self.nv, self.K, self.V), dtype=dt)
        for s in (range(self.max_slots) if slots is None else slots):
            pool[s] = self.state_slot(s)
        return pool

    def live_slots(self):
        return sorted(int(s) for s in self.slot_idx if s >= 0)


def _qkv(rng, T, nk, nv, K, V):
    return rng.standard_normal((T, 2 * nk * K + nv * V), dtype=np.float32)


def tiny(seed: int = 0) -> Workload:
    """batch=2 ragged rows of length 5 and 3, nk=1, nv=2, K=V=16, fp32 pool [4,2,16,16]."""
    rng = np.random.default_rng(seed)
    nk, nv, K, V = 1, 2, 16, 16
    offsets = np.array([0, 5, 8], dtype=np.int32)
    T = 8
    qkv = _qkv(rng, T, nk, nv, K, V)
    decay = rng.uniform(0.8, 1.0, (T, nv)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, (T, nv)).astype(np.float32)
    return Workload("tiny", nk, nv, K, V, qkv, decay, beta,
                    np.array([2, 0], dtype=np.int32), offsets, 4, "f32", seed, 0.1)


def decode(seed: int = 1, batch: int = 256, max_slots: int = 512, n_pad: int = 8,
           nk: int = 16, nv: int = 32, K: int = 128, state_dtype: str = "bf16") -> Workload:
    """One token per row; slot_idx a random permutation prefix with n_pad rows set to -1."""
    rng = np.random.default_rng(seed)
    V = K
    T = batch
    qkv = _qkv(rng, T, nk, nv, K, V)
    decay = rng.uniform(0.9, 1.0, (T, nv)).astype(np.float32)
    beta = _sigmoid(rng.standard_normal((T, nv))).astype(np.float32)
    slot_idx = rng.permutation(max_slots)[:batch].astype(np.int32)
    if n_pad:
        slot_idx[rng.choice(batch, size=n_pad, replace=False)] = -1
    offsets = np.arange(batch + 1, dtype=np.int32)
    return Workload("decode", nk, nv, K, V, qkv, decay, beta, slot_idx, offsets,
                    max_slots, state_dtype, seed, 0.05)


def prefill(seed: int = 2, batch: int = 8, max_slots: int = 16, lmin: int = 512,
            lmax: int = 4096, nk: int = 16, nv: int = 32, K: int = 128,
            state_dtype: str = "bf16", lengths=None, V: int = 0) -> Workload:
    """Ragged rows with lengths ~ U{lmin..lmax}; the pool is read and written in
    place; value head size V (K if 0)."""
    rng = np.random.default_rng(seed)
    V = V or K
    L = (np.asarray(lengths, dtype=np.int64) if lengths is not None
         else rng.integers(lmin, lmax + 1, size=batch))
    batch = len(L)
    offsets = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    T = int(offsets[-1])
    qkv = _qkv(rng, T, nk, nv, K, V)
    decay = rng.uniform(0.9, 1.0, (T, nv)).astype(np.float32)
    beta = _sigmoid(rng.standard_normal((T, nv))).astype(np.float32)
    slot_idx = rng.permutation(max_slots)[:batch].astype(np.int32)
    return Workload("prefill", nk, nv, K, V, qkv, decay, beta, slot_idx, offsets,
                    max_slots, state_dtype, seed, 0.05)


def verify_fold(seed: int = 3, batch: int = 128, draft: int = 5, long_len: int = 12,
                ring_len: int = 8, max_slots: int = 256, ring_rows: int = 256,
                nk: int = 16, nv: int = 32, K: int = 128, state_dtype: str = "bf16") -> Workload:
    """batch-1 rows of `draft` tokens plus a last row of `long_len` tokens; accepted
    counts ~ U{0..draft}; the long row gets count = its length (the fold skips it)."""
    rng = np.random.default_rng(seed)
    V = K
    L = np.full(batch, draft, dtype=np.int64)
    L[-1] = long_len
    offsets = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    T = int(offsets[-1])
    qkv = _qkv(rng, T, nk, nv, K, V)
    decay = rng.uniform(0.9, 1.0, (T, nv)).astype(np.float32)
    beta = _sigmoid(rng.standard_normal((T, nv))).astype(np.float32)
    slot_idx = rng.permutation(max_slots)[:batch].astype(np.int32)
    ring_slot_idx = rng.permutation(ring_rows)[:batch].astype(np.int32)
    counts = rng.integers(0, draft + 1, size=batch).astype(np.int32)
    counts[-1] = long_len
    return Workload("verify_fold", nk, nv, K, V, qkv, decay, beta, slot_idx, offsets,
                    max_slots, state_dtype, seed, 0.05, ring_len=ring_len,
                    ring_rows=ring_rows, ring_slot_idx=ring_slot_idx, counts=counts)


def gdp_snapshots(seed: int = 4, batch: int = 64, drafts: int = 4, householder: int = 2,
                  max_slots: int = 128, nk: int = 16, nv: int = 32, K: int = 128,
                  state_dtype: str = "f32", beta_per_value: bool = False) -> Workload:
    """Gated Delta Product spec-decode: `drafts` draft tokens x `householder` copies folded
    into the sequence ("core.ssm.ops.gdp.fused_recurrent", module summary): each step has
    its own k, v, beta and q; the log decay g ~ U(-0.1, 0) sits on the first copy of a
    draft token and g = 0 on the others.  steps_per_token = householder.  beta is
    head-wise, or per value element when beta_per_value."""
    rng = np.random.default_rng(seed)
    V = K
    Lr = drafts * householder
    offsets = (np.arange(batch + 1) * Lr).astype(np.int32)
    T = batch * Lr
    qkv = _qkv(rng, T, nk, nv, K, V)
    g = rng.uniform(-0.1, 0.0, (T, nv)).astype(np.float32)
    step_in_row = np.arange(T) % Lr
    g[(step_in_row % householder) != 0] = 0.0
    beta = _sigmoid(rng.standard_normal((T, nv, V) if beta_per_value else (T, nv))).astype(np.float32)
    slot_idx = rng.permutation(max_slots)[:batch].astype(np.int32)
    accepted = rng.integers(0, drafts, size=batch).astype(np.int32)
    return Workload("gdp_snapshots", nk, nv, K, V, qkv, g, beta, slot_idx, offsets,
                    max_slots, state_dtype, seed, 0.05, decay_is_log=True,
                    steps_per_token=householder, n_inter=drafts, accepted=accepted,
                    meta={"drafts": drafts, "householder": householder})


def random_case(seed: int, lengths, nk: int, nv: int, K: int, max_slots: int,
                state_dtype: str = "f32", n_pad: int = 0, decay_is_log: bool = False,
                use_l2norm: bool = True, scale: float = 0.0, state_std: float = 0.1,
                beta_per_value: bool = False, V: int = 0) -> Workload:
    """A small general case for parity tests: given row lengths, random slots;
    beta per value element when beta_per_value; value head size V (K if 0)."""
    rng = np.random.default_rng(seed)
    V = V or K
    L = np.asarray(lengths, dtype=np.int64)
    batch = len(L)
    offsets = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    T = int(offsets[-1])
    qkv = _qkv(rng, T, nk, nv, K, V)
    if decay_is_log:
        decay = rng.uniform(-0.1, 0.0, (T, nv)).astype(np.float32)
    else:
        decay = rng.uniform(0.8, 1.0, (T, nv)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, (T, nv, V) if beta_per_value else (T, nv)).astype(np.float32)
    slot_idx = rng.permutation(max_slots)[:batch].astype(np.int32)
    if n_pad:
        slot_idx[rng.choice(batch, size=n_pad, replace=False)] = -1
    return Workload(f"random{seed}", nk, nv, K, V, qkv, decay, beta, slot_idx, offsets,
                    max_slots, state_dtype, seed, state_std, decay_is_log=decay_is_log,
                    use_l2norm=use_l2norm, scale=scale)


@dataclass
class ConvInputs:
    """Pass-1 convolution parameters for a workload: weight [C, width], bias [C]
    (or None), conv-state pool [slots, C, width-1] (None for width 1)."""
    weight: np.ndarray
    bias: Optional[np.ndarray]
    state: Optional[np.ndarray]
    silu: bool


def conv_inputs(w: Workload, width: int = 4, seed: int = 0, bias: bool = True, silu: bool = True,
                weight_std: float = 0.5) -> ConvInputs:
    """Seeded Pass-1 convolution parameters for workload w: taps ~ N(0, weight_std^2),
    bias ~ N(0, 0.1^2), conv state ~ N(0, 1) (the raw inputs' scale)."""
    rng = np.random.default_rng([seed, 4049, width])
    C = w.qkv.shape[1]
    wt = (rng.standard_normal((C, width), dtype=np.float32) * np.float32(weight_std))
    b = rng.standard_normal(C, dtype=np.float32) * np.float32(0.1) if bias else None
    st = rng.standard_normal((w.max_slots, C, width - 1), dtype=np.float32) if width > 1 else None
    return ConvInputs(wt, b, st, silu)


CONFIGS = {
    "tiny": tiny,
    "decode": decode,
    "prefill": prefill,
    "verify_fold": verify_fold,
    "gdp_snapshots": gdp_snapshots,
}
