"""CPU oracle for the gated delta rule recurrence -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never does, and shares no code with it.

The arithmetic lives in ``gdr_oracle.c`` / ``gdr_oracle_core.h`` (plain C
loops, float64 by default, float32 on request), built here with gcc at -O2
and -ffp-contract=off.  This module is marshalling only: numpy arrays in,
numpy arrays out.  ``brute.py`` holds an independent numpy restatement of the
matrix form used to pin the C loops on tiny cases.

Arrays are dense and follow the pages' layouts:
  qkv    [T, 2*nk*K + nv*V] float32   ("gated_delta_recurrence_fwd_gpu", Args)
  decay  [T, nv] float32 (alpha, or log decay g when decay_is_log)
  beta   [T, nv] float32 (head-wise) or [T, nv, V] (per value element)
  state  [max_slots, nv, K, V] float32, or uint16 holding bfloat16 bits
  slot_idx [batch] int32 (-1 = padding), offsets [batch+1] int32
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "gdr_oracle.c"), os.path.join(_HERE, "gdr_oracle_core.h")]
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc if it is missing or older than its sources."""
    stale = force or not os.path.exists(_LIB_PATH) or any(
        os.path.getmtime(s) > os.path.getmtime(_LIB_PATH) for s in _SRC)
    if stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC[0], "-lm"]
        subprocess.run(cmd, check=True, cwd=_HERE)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("nv", ctypes.c_int32), ("nk", ctypes.c_int32),
        ("K", ctypes.c_int32), ("V", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64),
        ("qkv", ctypes.c_void_p), ("decay", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("decay_is_log", ctypes.c_int32), ("use_l2norm", ctypes.c_int32),
        ("scale", ctypes.c_double), ("eps", ctypes.c_double),
        ("state", ctypes.c_void_p), ("state_bf16", ctypes.c_int32),
        ("max_slots", ctypes.c_int64),
        ("slot_idx", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
        ("beta_per_value", ctypes.c_int32),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Problem)
            vp, i32 = ctypes.c_void_p, ctypes.c_int
            for prec in ("f64", "f32"):
                getattr(lib, f"oracle_fwd_{prec}").argtypes = [P, vp]
                getattr(lib, f"oracle_verify_ring_{prec}").argtypes = [P, vp, vp, i32, i32, i32, i32, vp]
                getattr(lib, f"oracle_fwd_snapshots_{prec}").argtypes = [P, vp, vp, i32, i32]
                getattr(lib, f"oracle_fold_{prec}").argtypes = [P, vp, i32, i32, i32, i32, vp, vp]
            lib.oracle_rollback.argtypes = [P, vp, i32, vp]
            i64 = ctypes.c_int64
            lib.oracle_conv1d.argtypes = [i32, i64, i32, i32, vp, vp, vp, i32, vp, i64, vp, vp, vp]
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_ring_record_elements.argtypes = [i32, i32, i32]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


class Problem:
    """Dense inputs of one call; ``state`` is modified in place by the passes."""

    def __init__(self, qkv, decay, beta, state, slot_idx, offsets, *, nk, nv, K, V,
                 decay_is_log=False, use_l2norm=True, scale=0.0, eps=1e-6):
        self.qkv = _c(qkv, np.float32)
        self.decay = _c(decay, np.float32)
        self.beta = _c(beta, np.float32)
        if state.dtype not in (np.float32, np.uint16):
            raise TypeError("state must be float32 or uint16 (bfloat16 bits)")
        if not state.flags.c_contiguous:
            raise ValueError("state must be C-contiguous (it is updated in place)")
        self.state = state
        self.slot_idx = _c(slot_idx, np.int32)
        self.offsets = _c(offsets, np.int32)
        self.nk, self.nv, self.K, self.V = int(nk), int(nv), int(K), int(V)
        self.decay_is_log, self.use_l2norm = bool(decay_is_log), bool(use_l2norm)
        self.scale, self.eps = float(scale), float(eps)
        T = self.qkv.shape[0] if self.qkv.ndim == 2 else 0
        self.total_tokens = T
        assert self.qkv.shape == (T, 2 * nk * K + nv * V), self.qkv.shape
        assert self.decay.shape == (T, nv)
        # beta: head-wise [T, nv] or per value element [T, nv, V]
        assert self.beta.shape in ((T, nv), (T, nv, V)), self.beta.shape
        self.beta_per_value = self.beta.ndim == 3
        assert state.ndim == 4 and state.shape[1:] == (nv, K, V), state.shape
        assert self.offsets.shape == (self.slot_idx.shape[0] + 1,)

    def _c_struct(self):
        return _Problem(
            batch=self.slot_idx.shape[0], nv=self.nv, nk=self.nk, K=self.K, V=self.V,
            total_tokens=self.total_tokens, qkv=_ptr(self.qkv), decay=_ptr(self.decay),
            beta=_ptr(self.beta), decay_is_log=int(self.decay_is_log),
            use_l2norm=int(self.use_l2norm), scale=self.scale, eps=self.eps,
            state=_ptr(self.state), state_bf16=int(self.state.dtype == np.uint16),
            max_slots=self.state.shape[0], slot_idx=_ptr(self.slot_idx),
            offsets=_ptr(self.offsets), beta_per_value=int(self.beta_per_value))

    def _out(self):
        return np.zeros((self.total_tokens, self.nv * self.V), dtype=np.float64)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


def fwd(p: Problem, work: str = "f64") -> np.ndarray:
    """Forward pass; returns out [T, nv*V] (float64) and advances p.state in place."""
    lib = _load()
    out = p._out()
    s = p._c_struct()
    _check(getattr(lib, f"oracle_fwd_{work}")(ctypes.byref(s), _ptr(out)), "fwd")
    return out


def fwd_dense(qkv, decay, beta, offsets, initial_state, *, nk, nv, K, V, state_dtype="f32",
              decay_is_log=False, use_l2norm=True, scale=0.0, eps=1e-6, work: str = "f64"):
    """Forward pass with a dense start state ("core.ssm.ops.gdp.fused_recurrent",
    initial_state [N, HV, K, V] or None for zeros, output_final_state): sequence n
    starts from initial_state[n] and its final state is returned in a new
    [N, HV, K, V] array (an empty sequence returns its initial state).  The
    gather/scatter around the recurrence, written out: sequence n runs on slot n
    of a pool that holds a copy of the start states.  Returns (out, final)."""
    N = len(offsets) - 1
    dt = np.uint16 if state_dtype == "bf16" else np.float32
    pool = (np.zeros((N, nv, K, V), dt) if initial_state is None
            else np.ascontiguousarray(initial_state, dtype=dt).copy())
    assert pool.shape == (N, nv, K, V)
    p = Problem(qkv, decay, beta, pool, np.arange(N, dtype=np.int32), offsets, nk=nk, nv=nv,
                K=K, V=V, decay_is_log=decay_is_log, use_l2norm=use_l2norm, scale=scale, eps=eps)
    out = fwd(p, work)
    return out, pool


def verify_ring(p: Problem, ring: np.ndarray, ring_slot_idx, ring_len: int,
                work: str = "f64") -> np.ndarray:
    """Verify pass; writes records into ``ring`` [ring_rows, nk, ring_len, stride],
    float32 or uint16 (bfloat16 bits, rounded to nearest-even)."""
    lib = _load()
    assert ring.dtype in (np.float32, np.uint16) and ring.flags.c_contiguous and ring.ndim == 4
    assert ring.shape[1] == p.nk and ring.shape[2] == ring_len
    rsi = _c(ring_slot_idx, np.int32)
    out = p._out()
    s = p._c_struct()
    _check(getattr(lib, f"oracle_verify_ring_{work}")(
        ctypes.byref(s), _ptr(out), _ptr(ring), int(ring.dtype == np.uint16), ring.shape[0],
        ring_len, ring.shape[3], _ptr(rsi)), "verify_ring")
    return out


def fold(p: Problem, ring: np.ndarray, ring_slot_idx, counts, ring_len: int,
         work: str = "f64") -> None:
    """Fold the first counts[b] records of each row into p.state in place; the ring
    is float32 or uint16 (bfloat16 bits)."""
    lib = _load()
    ring = _c(ring, np.uint16 if ring.dtype == np.uint16 else np.float32)
    rsi = _c(ring_slot_idx, np.int32)
    cnt = _c(counts, np.int32)
    s = p._c_struct()
    _check(getattr(lib, f"oracle_fold_{work}")(
        ctypes.byref(s), _ptr(ring), int(ring.dtype == np.uint16), ring.shape[0], ring_len,
        ring.shape[3], _ptr(rsi), _ptr(cnt)), "fold")


def fwd_snapshots(p: Problem, inter: np.ndarray, steps_per_token: int,
                  work: str = "f64") -> np.ndarray:
    """Forward pass that also stores inter[slot, i] after every steps_per_token steps."""
    lib = _load()
    assert inter.dtype == p.state.dtype and inter.flags.c_contiguous and inter.ndim == 5
    out = p._out()
    s = p._c_struct()
    _check(getattr(lib, f"oracle_fwd_snapshots_{work}")(
        ctypes.byref(s), _ptr(out), _ptr(inter), inter.shape[1], steps_per_token),
        "fwd_snapshots")
    return out


def rollback(p: Problem, inter: np.ndarray, accepted) -> None:
    """state[slot] <- inter[slot, accepted[b]] for every live row with accepted >= 0."""
    lib = _load()
    acc = _c(accepted, np.int32)
    s = p._c_struct()
    _check(lib.oracle_rollback(ctypes.byref(s), _ptr(inter), inter.shape[1], _ptr(acc)),
           "rollback")


def conv1d(x, weight, bias, silu: bool, conv_state, slot_idx, offsets) -> np.ndarray:
    """Pass-1 causal depthwise convolution ("gated_delta_recurrence_fwd_gpu",
    Args: qkv_conv_output is its output): x [T, C] float32, weight [C, W],
    bias [C] or None, SiLU or none; conv_state [slots, C, W-1] float32 is read
    at slot_idx and updated in place (None when W == 1).  Returns the float32
    output [T, C] (the readings are listed in gdr_oracle.c)."""
    lib = _load()
    x = _c(x, np.float32)
    weight = _c(weight, np.float32)
    C, Wd = weight.shape
    T = x.shape[0]
    assert x.shape == (T, C)
    b = None if bias is None else _c(bias, np.float32)
    if conv_state is not None:
        assert conv_state.dtype == np.float32 and conv_state.flags.c_contiguous
        assert conv_state.shape[1:] == (C, Wd - 1)
        slots = conv_state.shape[0]
    else:
        assert Wd == 1
        slots = 1 << 30
    si = _c(slot_idx, np.int32)
    off = _c(offsets, np.int32)
    y = np.zeros((T, C), np.float32)
    _check(lib.oracle_conv1d(si.shape[0], T, C, Wd, _ptr(x), _ptr(weight), _ptr(b), int(bool(silu)),
                             _ptr(conv_state), slots, _ptr(si), _ptr(off), _ptr(y)), "conv1d")
    return y


def fwd_conv(p: Problem, weight, bias, silu: bool, conv_state, work: str = "f64") -> np.ndarray:
    """The forward pass on Pass-1 output: p.qkv holds the RAW convolution input;
    the convolution (conv1d, conv_state updated in place) produces
    qkv_conv_output, which the recurrence then reads.  Returns out [T, nv*V]."""
    y = conv1d(p.qkv, weight, bias, silu, conv_state, p.slot_idx, p.offsets)
    q = Problem(y, p.decay, p.beta, p.state, p.slot_idx, p.offsets, nk=p.nk, nv=p.nv, K=p.K, V=p.V,
                decay_is_log=p.decay_is_log, use_l2norm=p.use_l2norm, scale=p.scale, eps=p.eps)
    return fwd(q, work)


def round_bf16(x) -> np.ndarray:
    """bfloat16 bits (uint16) of each value, rounded to nearest-even from float64."""
    lib = _load()
    flat = np.asarray(x, dtype=np.float64).ravel()
    return np.array([lib.oracle_round_bf16(float(v)) for v in flat],
                    dtype=np.uint16).reshape(np.shape(x))


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bfloat16 bits to float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ring_record_elements(K: int, V: int, ratio: int) -> int:
    return int(_load().oracle_ring_record_elements(K, V, ratio))
