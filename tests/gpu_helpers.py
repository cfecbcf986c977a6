"""Helpers for GPU tests: move a seeded workload to the device, run the C ABI
through the binding, and bring results back as numpy for comparison."""
from __future__ import annotations

import numpy as np
import torch

import gated_deltanet_linear_gdr_gb300 as gdr
from gated_deltanet_linear_gdr_gb300 import workloads as W

DEV = torch.device("cuda:0")

OUT_ATOL = 2e-3        # outputs: max abs error (stated tolerance of the path)
F32_STATE_TOL = 1e-4   # float32 state/snapshots: abs, and rel where |ref| > 1e-3


def pool_to_dev(pool: np.ndarray) -> torch.Tensor:
    if pool.dtype == np.uint16:
        return torch.from_numpy(pool.view(np.int16).copy()).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(pool.copy()).to(DEV)


def pool_to_host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def as_f64(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


class Dev:
    """Device copies of a workload's per-call inputs."""

    def __init__(self, w: W.Workload, pool: np.ndarray):
        self.w = w
        self.qkv = torch.from_numpy(w.qkv).to(DEV)
        self.decay = torch.from_numpy(w.decay).to(DEV)
        self.beta = torch.from_numpy(w.beta).to(DEV)
        self.slot = torch.from_numpy(w.slot_idx).to(DEV)
        self.off = torch.from_numpy(w.offsets).to(DEV)
        self.state = pool_to_dev(pool)
        self.kw = dict(decay_is_log=w.decay_is_log, use_qk_l2norm=w.use_l2norm, scale=w.scale,
                       eps=w.eps)

    def fwd(self, max_row_len=0, out=None):
        return gdr.gdr_fwd(self.qkv, self.decay, self.beta, self.state, self.slot, self.off,
                           out=out, max_row_len=max_row_len, **self.kw)

    def verify(self, ring, ring_slot, max_row_len=0, out=None):
        return gdr.gdr_verify_ring(self.qkv, self.decay, self.beta, self.state, self.slot,
                                   self.off, ring, ring_slot, out=out, max_row_len=max_row_len, **self.kw)

    def snapshots(self, inter, spt, max_row_len=0, out=None):
        return gdr.gdr_fwd_snapshots(self.qkv, self.decay, self.beta, self.state, self.slot,
                                     self.off, inter, spt, out=out, max_row_len=max_row_len, **self.kw)


def check_out(gpu_out: torch.Tensor, ref: np.ndarray, atol=OUT_ATOL):
    got = gpu_out.detach().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= atol, f"max |out - oracle| = {err:.3e} > {atol}"
    return err


def check_state(gpu_state: np.ndarray, ref_state: np.ndarray, slots=None):
    """bf16: within one bf16 ulp of the oracle's value (floor 2^-10); f32: 1e-4 abs/rel."""
    sl = slice(None) if slots is None else list(slots)
    g, r = gpu_state[sl], ref_state[sl]
    if g.dtype == np.uint16:
        gf, rf = as_f64(g), as_f64(r)
        mag = np.maximum(np.abs(rf), 2.0 ** -10)
        ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
        bad = np.abs(gf - rf) > ulp
        assert not bad.any(), f"{int(bad.sum())} bf16 state entries beyond 1 ulp"
    else:
        gf, rf = g.astype(np.float64), r.astype(np.float64)
        diff = np.abs(gf - rf)
        assert diff.max() <= F32_STATE_TOL, f"max abs state error {diff.max():.3e}"
        big = np.abs(rf) > 1e-3
        if big.any():
            rel = (diff[big] / np.abs(rf[big])).max()
            assert rel <= F32_STATE_TOL, f"max rel state error {rel:.3e}"


def ring_for(w: W.Workload, ring_len: int, rows: int, dtype=torch.float32) -> torch.Tensor:
    stride = gdr.gdr_ring_record_elements(w.K, w.V, w.nv // w.nk)
    stride = (stride + 7) // 8 * 8
    return torch.full((rows, w.nk, ring_len, stride), float("nan"), dtype=dtype, device=DEV)


def ring_to_host(t: torch.Tensor) -> np.ndarray:
    """float32 ring as float32, bfloat16 ring as its uint16 bits."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def ring_to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(a.copy()).to(DEV)
