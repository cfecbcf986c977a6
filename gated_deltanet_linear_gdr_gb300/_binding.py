"""Thin ctypes binding over libgdr.so (include/gdr.h).

Argument marshalling only: tensors are checked for dtype/device/shape, their
data pointers and strides are packed into gdr_step_args, and the C entry point
of the same name runs every step of the path on the GPU.  PyTorch supplies the
device memory and the current stream; nothing here computes.

If libgdr.so is missing the first call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdr.so")

GDR_OK, GDR_ERR_INVALID_ARG, GDR_ERR_UNSUPPORTED, GDR_ERR_CUDA = 0, -1, -2, -3
GDR_F32, GDR_BF16 = 0, 1
STATUS_BITS = {
    0x1: "BAD_SLOT", 0x2: "BAD_OFFSETS", 0x4: "BAD_RING_SLOT", 0x8: "BAD_COUNT",
    0x10: "ROW_TOO_LONG", 0x20: "BAD_ACCEPTED", 0x40: "SNAPSHOT_OVERFLOW",
}


class GdrError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"gdr error {code}: {msg}")
        self.code = code


class gdr_host_io(ctypes.Structure):
    """Mirror of struct gdr_host_io in include/gdr.h (host pointers)."""
    _fields_ = [
        ("qkv", ctypes.c_void_p), ("decay", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("slot_idx", ctypes.c_void_p), ("offsets", ctypes.c_void_p), ("out", ctypes.c_void_p),
    ]


class gdr_step_args(ctypes.Structure):
    """Mirror of struct gdr_step_args in include/gdr.h (same order and types)."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("nv", ctypes.c_int32), ("nk", ctypes.c_int32),
        ("K", ctypes.c_int32), ("V", ctypes.c_int32),
        ("decay_is_log", ctypes.c_int32), ("use_qk_l2norm", ctypes.c_int32),
        ("state_dtype", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64), ("max_row_len", ctypes.c_int64),
        ("qkv", ctypes.c_void_p), ("qkv_seq_stride", ctypes.c_int64),
        ("qkv_chan_stride", ctypes.c_int64),
        ("decay", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("tok_seq_stride", ctypes.c_int64), ("tok_head_stride", ctypes.c_int64),
        ("scale", ctypes.c_float), ("eps", ctypes.c_float),
        ("out", ctypes.c_void_p), ("out_seq_stride", ctypes.c_int64),
        ("out_vdim_stride", ctypes.c_int64),
        ("state", ctypes.c_void_p), ("state_slot_stride", ctypes.c_int64),
        ("state_head_stride", ctypes.c_int64), ("state_kdim_stride", ctypes.c_int64),
        ("state_vdim_stride", ctypes.c_int64), ("max_slots", ctypes.c_int64),
        ("slot_idx", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
        ("beta_seq_stride", ctypes.c_int64), ("beta_head_stride", ctypes.c_int64),
        ("beta_vdim_stride", ctypes.c_int64),
    ]


class gdr_conv_args(ctypes.Structure):
    """Mirror of struct gdr_conv_args in include/gdr.h."""
    _fields_ = [
        ("width", ctypes.c_int32), ("activation", ctypes.c_int32),
        ("weight", ctypes.c_void_p), ("weight_chan_stride", ctypes.c_int64),
        ("weight_tap_stride", ctypes.c_int64), ("bias", ctypes.c_void_p),
        ("conv_state", ctypes.c_void_p), ("state_slot_stride", ctypes.c_int64),
        ("state_chan_stride", ctypes.c_int64), ("state_tap_stride", ctypes.c_int64),
    ]


_lock = threading.Lock()
_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libgdr.so (built by gated_deltanet_linear_gdr_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"{p} is missing: build it with `python -c \"import __graft_entry__ as g; "
                    f"g.build()\"` (the GDR path has no CPU or Python fallback)")
            lib = ctypes.CDLL(p)
            A = ctypes.POINTER(gdr_step_args)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            sig = {
                "gdr_last_error": ([], ctypes.c_char_p),
                "gdr_version": ([], ctypes.c_int),
                "gdr_output_shape": ([i64, i32, i32, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
                "gdr_ring_record_elements": ([i32, i32, i32], ctypes.c_int),
                "gdr_fwd": ([A, vp], ctypes.c_int),
                "gdr_fwd_host": ([A, ctypes.POINTER(gdr_host_io), i32, vp, vp, vp], ctypes.c_int),
                "gdr_fwd_host_noalloc": ([A, ctypes.POINTER(gdr_host_io), i32, vp, vp, vp], ctypes.c_int),
                "gdr_fwd_dense": ([A, vp, vp, vp], ctypes.c_int),
                "gdr_fwd_conv": ([A, ctypes.POINTER(gdr_conv_args), vp], ctypes.c_int),
                "gdr_verify_ring": ([A, vp, i32, i64, i32, i64, vp, vp], ctypes.c_int),
                "gdr_fold": ([A, vp, i32, i64, i32, i64, vp, vp, vp], ctypes.c_int),
                "gdr_fwd_snapshots": ([A, vp, i64, i64, i64, i32, i32, vp], ctypes.c_int),
                "gdr_rollback": ([A, vp, i64, i64, i64, i32, vp, vp], ctypes.c_int),
                "gdr_get_status": ([ctypes.POINTER(ctypes.c_uint32), i32], ctypes.c_int),
                "gdr_probe_fma": ([i32, i32, i32, vp, i64, ctypes.POINTER(ctypes.c_int32), vp], ctypes.c_int),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            if path is None:
                _lib = lib
            else:
                return lib
    return _lib


def _check(rc: int):
    if rc != GDR_OK:
        msg = load_library().gdr_last_error().decode(errors="replace")
        raise GdrError(rc, msg)


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return t


def _ring_dtype(ring: torch.Tensor) -> int:
    return GDR_BF16 if ring.dtype == torch.bfloat16 else GDR_F32


def _state_dtype(state: torch.Tensor) -> int:
    if state.dtype == torch.bfloat16:
        return GDR_BF16
    if state.dtype == torch.float32:
        return GDR_F32
    raise TypeError(f"state dtype {state.dtype}: expected bfloat16 or float32")


def make_args(qkv, decay, beta, state, slot_idx, offsets, out, *, nk: int,
              decay_is_log=False, use_qk_l2norm=True, scale=0.0, eps=1e-6,
              max_row_len=0) -> gdr_step_args:
    """Pack tensors into gdr_step_args (no copies; strides passed through)."""
    _dev(state, "state", (torch.bfloat16, torch.float32))
    if state.dim() != 4:
        raise ValueError("state must be [max_slots, nv, K, V]")
    max_slots, nv, K, V = state.shape
    _dev(slot_idx, "slot_idx", torch.int32)
    batch = slot_idx.shape[0]
    a = gdr_step_args()
    a.batch, a.nv, a.nk, a.K, a.V = batch, nv, nk, K, V
    a.decay_is_log, a.use_qk_l2norm = int(bool(decay_is_log)), int(bool(use_qk_l2norm))
    a.state_dtype = _state_dtype(state)
    a.max_row_len = int(max_row_len)
    a.scale, a.eps = float(scale), float(eps)
    a.state = state.data_ptr()
    (a.state_slot_stride, a.state_head_stride, a.state_kdim_stride,
     a.state_vdim_stride) = state.stride()
    a.max_slots = max_slots
    a.slot_idx = slot_idx.data_ptr()
    if qkv is not None:
        _dev(qkv, "qkv", torch.float32)
        _dev(decay, "decay", torch.float32)
        _dev(beta, "beta", torch.float32)
        _dev(out, "out", torch.float32)
        _dev(offsets, "offsets", torch.int32)
        T = qkv.shape[0]
        if qkv.shape[1] != 2 * nk * K + nv * V:
            raise ValueError(f"qkv has {qkv.shape[1]} channels, expected 2*nk*K + nv*V = "
                             f"{2 * nk * K + nv * V}")
        if decay.shape != (T, nv):
            raise ValueError("decay must be [T, nv]")
        if beta.shape == (T, nv, V):
            # per value element ("core.ssm.ops.gdp.fused_recurrent", beta [B, T, HV, V])
            a.beta_seq_stride, a.beta_head_stride, a.beta_vdim_stride = beta.stride()
            if a.beta_vdim_stride <= 0:
                raise ValueError("per-element beta needs a positive value-dim stride")
        elif beta.shape != (T, nv) or decay.stride() != beta.stride():
            raise ValueError("beta must be [T, nv] with decay's strides, or [T, nv, V]")
        if out.shape != (T, nv * V):
            raise ValueError(f"out must be [T, nv*V] = [{T}, {nv * V}]")
        if offsets.shape != (batch + 1,) or not offsets.is_contiguous():
            raise ValueError("offsets must be a contiguous [batch+1] int32 tensor")
        a.total_tokens = T
        a.qkv = qkv.data_ptr()
        a.qkv_seq_stride, a.qkv_chan_stride = qkv.stride()
        a.decay, a.beta = decay.data_ptr(), beta.data_ptr()
        a.tok_seq_stride, a.tok_head_stride = decay.stride()
        a.out = out.data_ptr()
        a.out_seq_stride, a.out_vdim_stride = out.stride()
        a.offsets = offsets.data_ptr()
    if not slot_idx.is_contiguous():
        raise ValueError("slot_idx must be contiguous")
    return a


def _nk_from_qkv(qkv, state):
    nv, K, V = state.shape[1:]
    rest = qkv.shape[1] - nv * V
    if rest <= 0 or rest % (2 * K):
        raise ValueError("cannot infer nk from qkv channels")
    return rest // (2 * K)


def gdr_output_shape(total_tokens: int, nv: int, V: int):
    shp = (ctypes.c_int64 * 2)()
    _check(load_library().gdr_output_shape(total_tokens, nv, V, shp))
    return int(shp[0]), int(shp[1])


def gdr_ring_record_elements(K: int, V: int, ratio: int) -> int:
    n = load_library().gdr_ring_record_elements(K, V, ratio)
    if n < 0:
        _check(n)
    return n


def gdr_fwd(qkv, decay, beta, state, slot_idx, offsets, out=None, *, decay_is_log=False,
            use_qk_l2norm=True, scale=0.0, eps=1e-6, max_row_len=0):
    """Forward pass ("gated_delta_recurrence_fwd_gpu"); state updated in place; returns out."""
    if out is None:
        out = torch.empty(gdr_output_shape(qkv.shape[0], state.shape[1], state.shape[3]),
                          dtype=torch.float32, device=qkv.device)
    a = make_args(qkv, decay, beta, state, slot_idx, offsets, out, nk=_nk_from_qkv(qkv, state),
                  decay_is_log=decay_is_log, use_qk_l2norm=use_qk_l2norm, scale=scale, eps=eps,
                  max_row_len=max_row_len)
    _check(load_library().gdr_fwd(ctypes.byref(a), _stream(qkv.device)))
    return out


def _host(t: torch.Tensor, name: str, dtype):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) torch.Tensor")
    if t.dtype != dtype or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous {dtype} tensor")
    return t


class HostForward:
    """gdr_fwd_host for host-resident tokens: the forward pass
    ("gated_delta_recurrence_fwd_gpu") with the tokens copied in and the
    output copied back inside one C-ABI call, row groups pipelined over three
    streams (copies in, compute, copies out).

    Owns the device staging buffers for batches of up to `batch` rows and
    `total_tokens` tokens and the two side streams; the pool stays the
    caller's device tensor.  Host tensors should be pinned
    (tensor.pin_memory()) for the copies to overlap the compute."""

    def __init__(self, state, nk: int, batch: int, total_tokens: int, *, decay_is_log=False,
                 use_qk_l2norm=True, scale=0.0, eps=1e-6, max_row_len=0, chunks=0):
        _dev(state, "state", (torch.bfloat16, torch.float32))
        dev = state.device
        nv, K, V = state.shape[1:]
        f32, i32 = torch.float32, torch.int32
        self.state = state
        self.qkv = torch.empty((total_tokens, 2 * nk * K + nv * V), dtype=f32, device=dev)
        self.decay = torch.empty((total_tokens, nv), dtype=f32, device=dev)
        self.beta = torch.empty((total_tokens, nv), dtype=f32, device=dev)
        self.out = torch.empty((total_tokens, nv * V), dtype=f32, device=dev)
        self.slot_idx = torch.empty((batch,), dtype=i32, device=dev)
        self.offsets = torch.empty((batch + 1,), dtype=i32, device=dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.chunks = int(chunks)
        self.args = make_args(self.qkv, self.decay, self.beta, state, self.slot_idx, self.offsets, self.out,
                              nk=nk, decay_is_log=decay_is_log, use_qk_l2norm=use_qk_l2norm, scale=scale,
                              eps=eps, max_row_len=max_row_len)
        self.device = dev

    def __call__(self, qkv, decay, beta, slot_idx, offsets, out, stream: Optional[int] = None):
        """Runs the pass on host tensors; `out` (host, [T, nv*V]) holds the
        result once `stream` (default: the current stream) has passed the call."""
        for t, n, d in ((qkv, "qkv", torch.float32), (decay, "decay", torch.float32),
                        (beta, "beta", torch.float32), (slot_idx, "slot_idx", torch.int32),
                        (offsets, "offsets", torch.int32), (out, "out", torch.float32)):
            _host(t, n, d)
        if tuple(qkv.shape) != tuple(self.qkv.shape) or tuple(out.shape) != tuple(self.out.shape):
            raise ValueError("qkv / out shapes differ from the staging buffers")
        if slot_idx.shape[0] != self.slot_idx.shape[0] or offsets.shape[0] != self.offsets.shape[0]:
            raise ValueError("slot_idx / offsets lengths differ from the staging buffers")
        io = gdr_host_io(qkv.data_ptr(), decay.data_ptr(), beta.data_ptr(), slot_idx.data_ptr(),
                         offsets.data_ptr(), out.data_ptr())
        s = _stream(self.device) if stream is None else stream
        _check(load_library().gdr_fwd_host(ctypes.byref(self.args), ctypes.byref(io), self.chunks, s,
                                           self.h2d.cuda_stream, self.d2h.cuda_stream))
        return out


def make_conv_args(weight, bias, conv_state, state, activation="silu") -> gdr_conv_args:
    """Pack the Pass-1 convolution's tensors into gdr_conv_args: weight
    [conv_dim, width] float32, bias [conv_dim] float32 or None, conv_state
    [slots, conv_dim, width-1] float32 indexed like the pool `state` (None
    when width == 1); activation "silu" or None."""
    _dev(weight, "conv_weight", torch.float32)
    if weight.dim() != 2:
        raise ValueError("conv_weight must be [conv_dim, width]")
    C, width = weight.shape
    c = gdr_conv_args()
    c.width = width
    if activation not in (None, "silu"):
        raise ValueError('activation must be "silu" or None')
    c.activation = 1 if activation == "silu" else 0
    c.weight = weight.data_ptr()
    c.weight_chan_stride, c.weight_tap_stride = weight.stride()
    if bias is not None:
        _dev(bias, "conv_bias", torch.float32)
        if bias.shape != (C,) or bias.stride() != (1,):
            raise ValueError("conv_bias must be a contiguous [conv_dim] tensor")
        c.bias = bias.data_ptr()
    if width > 1:
        if conv_state is None:
            raise ValueError("conv_state is needed for width > 1")
        _dev(conv_state, "conv_state", torch.float32)
        if conv_state.dim() != 3 or conv_state.shape[1:] != (C, width - 1):
            raise ValueError(f"conv_state must be [slots, {C}, {width - 1}]")
        if conv_state.shape[0] < state.shape[0]:
            raise ValueError("conv_state needs one row per pool slot (it is indexed by slot_idx)")
        c.conv_state = conv_state.data_ptr()
        c.state_slot_stride, c.state_chan_stride, c.state_tap_stride = conv_state.stride()
    return c


def gdr_fwd_conv(x, decay, beta, state, slot_idx, offsets, conv_weight, conv_bias=None, conv_state=None,
                 activation="silu", out=None, *, decay_is_log=False, use_qk_l2norm=True, scale=0.0, eps=1e-6,
                 max_row_len=0):
    """Forward pass on the raw Pass-1 input x [T, 2*nk*K + nv*V]: the causal
    depthwise convolution ("gated_delta_recurrence_fwd_gpu", Args:
    qkv_conv_output is the Conv1d output from Pass 1) fused into the
    recurrence's operand staging; state and conv_state updated in place;
    returns out."""
    if out is None:
        out = torch.empty(gdr_output_shape(x.shape[0], state.shape[1], state.shape[3]),
                          dtype=torch.float32, device=x.device)
    a = make_args(x, decay, beta, state, slot_idx, offsets, out, nk=_nk_from_qkv(x, state),
                  decay_is_log=decay_is_log, use_qk_l2norm=use_qk_l2norm, scale=scale, eps=eps,
                  max_row_len=max_row_len)
    if conv_weight.shape[0] != x.shape[1]:
        raise ValueError("conv_weight must have one row per input channel")
    c = make_conv_args(conv_weight, conv_bias, conv_state, state, activation)
    _check(load_library().gdr_fwd_conv(ctypes.byref(a), ctypes.byref(c), _stream(x.device)))
    return out


def prepare_fwd_conv(x, decay, beta, state, slot_idx, offsets, conv_weight, conv_bias, conv_state, out, *,
                     activation="silu", decay_is_log=False, use_qk_l2norm=True, scale=0.0, eps=1e-6,
                     max_row_len=0) -> "Prepared":
    a = make_args(x, decay, beta, state, slot_idx, offsets, out, nk=_nk_from_qkv(x, state),
                  decay_is_log=decay_is_log, use_qk_l2norm=use_qk_l2norm, scale=scale, eps=eps,
                  max_row_len=max_row_len)
    c = make_conv_args(conv_weight, conv_bias, conv_state, state, activation)
    lib = load_library()
    return Prepared(lambda ap, cp, s: lib.gdr_fwd_conv(ap, cp, s), a, (ctypes.byref(c),),
                    (x, decay, beta, state, slot_idx, offsets, out, conv_weight, conv_bias, conv_state, c),
                    x.device)


def gdr_fwd_dense(qkv, decay, beta, offsets, initial_state=None, output_final_state=True, out=None, *,
                  nv=None, K=None, state_dtype=torch.float32, decay_is_log=False, use_qk_l2norm=True,
                  scale=0.0, eps=1e-6, max_row_len=0):
    """Forward pass with a dense start / end state ("core.ssm.ops.gdp.fused_recurrent",
    initial_state [N, HV, K, V] or None for zeros, output_final_state).  Returns
    (out, final_state); final_state is a new [N, HV, K, V] tensor of the start
    state's dtype (None unless output_final_state).  Without an initial state,
    nv and K (= V) give the shape and state_dtype the dtype."""
    batch = offsets.shape[0] - 1
    if initial_state is not None:
        ref = initial_state
    else:
        if nv is None or K is None:
            raise ValueError("without initial_state, nv and K are needed")
        ref = torch.empty((batch, nv, K, K), dtype=state_dtype, device=qkv.device)
    final = torch.empty_like(ref, memory_format=torch.contiguous_format) if output_final_state else None
    if initial_state is not None and final is not None and final.stride() != initial_state.stride():
        raise ValueError("initial_state must be contiguous (final_state shares its strides)")
    if out is None:
        out = torch.empty(gdr_output_shape(qkv.shape[0], ref.shape[1], ref.shape[3]),
                          dtype=torch.float32, device=qkv.device)
    rows = torch.zeros(batch, dtype=torch.int32, device=qkv.device)  # shape only: not read
    a = make_args(qkv, decay, beta, ref, rows, offsets, out, nk=_nk_from_qkv(qkv, ref),
                  decay_is_log=decay_is_log, use_qk_l2norm=use_qk_l2norm, scale=scale, eps=eps,
                  max_row_len=max_row_len)
    _check(load_library().gdr_fwd_dense(
        ctypes.byref(a), None if initial_state is None else initial_state.data_ptr(),
        None if final is None else final.data_ptr(), _stream(qkv.device)))
    return out, final


def gdr_verify_ring(qkv, decay, beta, state, slot_idx, offsets, ring, ring_slot_idx, out=None, *,
                    decay_is_log=False, use_qk_l2norm=True, scale=0.0, eps=1e-6, max_row_len=0):
    """Verify pass ("gated_delta_recurrence_verify_ring_gpu"); ring is
    [ring_rows, nk, ring_len, record_stride] float32 or bfloat16 (dense)."""
    _dev(ring, "ring", (torch.float32, torch.bfloat16))
    _dev(ring_slot_idx, "ring_slot_idx", torch.int32)
    if ring.dim() != 4 or not ring.is_contiguous():
        raise ValueError("ring must be a contiguous [ring_rows, nk, ring_len, record_stride] tensor")
    if out is None:
        out = torch.empty(gdr_output_shape(qkv.shape[0], state.shape[1], state.shape[3]),
                          dtype=torch.float32, device=qkv.device)
    nk = _nk_from_qkv(qkv, state)
    if ring.shape[1] != nk:
        raise ValueError("ring.shape[1] must equal nk")
    a = make_args(qkv, decay, beta, state, slot_idx, offsets, out, nk=nk, decay_is_log=decay_is_log,
                  use_qk_l2norm=use_qk_l2norm, scale=scale, eps=eps, max_row_len=max_row_len)
    _check(load_library().gdr_verify_ring(ctypes.byref(a), ring.data_ptr(), _ring_dtype(ring), ring.shape[0],
                                          ring.shape[2], ring.shape[3], ring_slot_idx.data_ptr(),
                                          _stream(qkv.device)))
    return out


def gdr_fold(state, slot_idx, ring, ring_slot_idx, counts):
    """Fold the first counts[b] records of each row into its slot (in place)."""
    _dev(ring, "ring", (torch.float32, torch.bfloat16))
    _dev(ring_slot_idx, "ring_slot_idx", torch.int32)
    _dev(counts, "counts", torch.int32)
    if ring.dim() != 4 or not ring.is_contiguous():
        raise ValueError("ring must be a contiguous [ring_rows, nk, ring_len, record_stride] tensor")
    a = make_args(None, None, None, state, slot_idx, None, None, nk=ring.shape[1])
    _check(load_library().gdr_fold(ctypes.byref(a), ring.data_ptr(), _ring_dtype(ring), ring.shape[0],
                                   ring.shape[2], ring.shape[3], ring_slot_idx.data_ptr(),
                                   counts.data_ptr(), _stream(state.device)))


def _inter_strides(inter, state):
    if inter.dtype != state.dtype:
        raise TypeError("intermediate_states must have the pool's dtype")
    if inter.dim() != 5 or inter.shape[2:] != state.shape[1:]:
        raise ValueError("intermediate_states must be [slots, n_inter, nv, K, V]")
    if inter.shape[0] < state.shape[0]:
        # the kernels index it by pool slot, which is only checked against the pool's slot count
        raise ValueError(f"intermediate_states has {inter.shape[0]} slot rows; it needs one per pool "
                         f"slot ({state.shape[0]})")
    K, V = state.shape[2:]
    if inter.stride(4) != 1 or inter.stride(3) != V:
        raise ValueError("each [K, V] block of intermediate_states must be dense")
    return inter.stride(0), inter.stride(1), inter.stride(2), inter.shape[1]


def gdr_fwd_snapshots(qkv, decay, beta, state, slot_idx, offsets, inter, steps_per_token, out=None,
                      *, decay_is_log=False, use_qk_l2norm=True, scale=0.0, eps=1e-6,
                      max_row_len=0):
    """Forward pass + snapshots ("core.ssm.ops.gdp.fused_recurrent", intermediate_states)."""
    _dev(inter, "intermediate_states")
    ss, st, sh, n_inter = _inter_strides(inter, state)
    if out is None:
        out = torch.empty(gdr_output_shape(qkv.shape[0], state.shape[1], state.shape[3]),
                          dtype=torch.float32, device=qkv.device)
    a = make_args(qkv, decay, beta, state, slot_idx, offsets, out, nk=_nk_from_qkv(qkv, state),
                  decay_is_log=decay_is_log, use_qk_l2norm=use_qk_l2norm, scale=scale, eps=eps,
                  max_row_len=max_row_len)
    _check(load_library().gdr_fwd_snapshots(ctypes.byref(a), inter.data_ptr(), ss, st, sh,
                                            n_inter, int(steps_per_token), _stream(qkv.device)))
    return out


def gdr_rollback(state, slot_idx, inter, accepted):
    """state[slot] <- intermediate_states[slot, accepted[b]] (in place)."""
    _dev(inter, "intermediate_states")
    _dev(accepted, "accepted", torch.int32)
    ss, st, sh, n_inter = _inter_strides(inter, state)
    a = make_args(None, None, None, state, slot_idx, None, None, nk=1)
    _check(load_library().gdr_rollback(ctypes.byref(a), inter.data_ptr(), ss, st, sh, n_inter,
                                       accepted.data_ptr(), _stream(state.device)))


def gdr_get_status(clear: bool = True) -> int:
    """Device status word (GDR_STATUS_* bits); synchronises the device."""
    v = ctypes.c_uint32(0)
    _check(load_library().gdr_get_status(ctypes.byref(v), int(bool(clear))))
    return int(v.value)


def gdr_probe_fma(pattern: int, warps_per_subpartition: int, iterations: int, sink: torch.Tensor) -> int:
    """Diagnostic FP32-pipe probe of include/gdr.h (pattern 0: the recurrence's
    per-element sweep; 1: packed FMAs with reusable operands; 2: with three
    distinct operands).  Launches on the current stream; returns the CTA count
    (one per SM, 128 * warps_per_subpartition threads each)."""
    _dev(sink, "sink", torch.float32)
    if not sink.is_contiguous():
        raise ValueError("sink must be contiguous")
    ctas = ctypes.c_int32(0)
    _check(load_library().gdr_probe_fma(int(pattern), int(warps_per_subpartition), int(iterations), sink.data_ptr(),
                                        sink.numel(), ctypes.byref(ctas), _stream(sink.device)))
    return int(ctas.value)


def status_names(bits: int):
    return [n for b, n in STATUS_BITS.items() if bits & b]


class Prepared:
    """A C-ABI call with its arguments marshalled once.

    Calling it re-issues the same entry point on the same device buffers with
    no per-call Python marshalling (the buffers' contents may change between
    calls; their addresses, shapes and strides may not).  Useful for repeated
    decode steps and for capturing the call into a CUDA graph."""

    def __init__(self, fn, args: gdr_step_args, extra, keep, device):
        self._fn = fn
        self._args = args
        self._extra = extra
        self._keep = keep  # tensors whose storage the call uses
        self._device = device

    def __call__(self, stream: Optional[int] = None):
        s = _stream(self._device) if stream is None else stream
        _check(self._fn(ctypes.byref(self._args), *self._extra, s))


def prepare_fwd(qkv, decay, beta, state, slot_idx, offsets, out, *, decay_is_log=False,
                use_qk_l2norm=True, scale=0.0, eps=1e-6, max_row_len=0) -> Prepared:
    a = make_args(qkv, decay, beta, state, slot_idx, offsets, out, nk=_nk_from_qkv(qkv, state),
                  decay_is_log=decay_is_log, use_qk_l2norm=use_qk_l2norm, scale=scale, eps=eps,
                  max_row_len=max_row_len)
    return Prepared(load_library().gdr_fwd, a, (),
                    (qkv, decay, beta, state, slot_idx, offsets, out), qkv.device)


def prepare_verify_ring(qkv, decay, beta, state, slot_idx, offsets, ring, ring_slot_idx, out, *,
                        decay_is_log=False, use_qk_l2norm=True, scale=0.0, eps=1e-6,
                        max_row_len=0) -> Prepared:
    _dev(ring, "ring", (torch.float32, torch.bfloat16))
    _dev(ring_slot_idx, "ring_slot_idx", torch.int32)
    if ring.dim() != 4 or not ring.is_contiguous():
        raise ValueError("ring must be a contiguous [ring_rows, nk, ring_len, record_stride] tensor")
    a = make_args(qkv, decay, beta, state, slot_idx, offsets, out, nk=_nk_from_qkv(qkv, state),
                  decay_is_log=decay_is_log, use_qk_l2norm=use_qk_l2norm, scale=scale, eps=eps,
                  max_row_len=max_row_len)
    extra = (ring.data_ptr(), _ring_dtype(ring), ring.shape[0], ring.shape[2], ring.shape[3],
             ring_slot_idx.data_ptr())
    return Prepared(load_library().gdr_verify_ring, a, extra,
                    (qkv, decay, beta, state, slot_idx, offsets, out, ring, ring_slot_idx),
                    qkv.device)


def prepare_fold(state, slot_idx, ring, ring_slot_idx, counts) -> Prepared:
    _dev(ring, "ring", (torch.float32, torch.bfloat16))
    _dev(ring_slot_idx, "ring_slot_idx", torch.int32)
    _dev(counts, "counts", torch.int32)
    if ring.dim() != 4 or not ring.is_contiguous():
        raise ValueError("ring must be a contiguous [ring_rows, nk, ring_len, record_stride] tensor")
    a = make_args(None, None, None, state, slot_idx, None, None, nk=ring.shape[1])
    extra = (ring.data_ptr(), _ring_dtype(ring), ring.shape[0], ring.shape[2], ring.shape[3],
             ring_slot_idx.data_ptr(), counts.data_ptr())
    return Prepared(load_library().gdr_fold, a, extra,
                    (state, slot_idx, ring, ring_slot_idx, counts), state.device)


def prepare_fwd_snapshots(qkv, decay, beta, state, slot_idx, offsets, inter, steps_per_token, out,
                          *, decay_is_log=False, use_qk_l2norm=True, scale=0.0, eps=1e-6,
                          max_row_len=0) -> Prepared:
    _dev(inter, "intermediate_states")
    ss, st, sh, n_inter = _inter_strides(inter, state)
    a = make_args(qkv, decay, beta, state, slot_idx, offsets, out, nk=_nk_from_qkv(qkv, state),
                  decay_is_log=decay_is_log, use_qk_l2norm=use_qk_l2norm, scale=scale, eps=eps,
                  max_row_len=max_row_len)
    extra = (inter.data_ptr(), ss, st, sh, n_inter, int(steps_per_token))
    return Prepared(load_library().gdr_fwd_snapshots, a, extra,
                    (qkv, decay, beta, state, slot_idx, offsets, out, inter), qkv.device)


def prepare_rollback(state, slot_idx, inter, accepted) -> Prepared:
    _dev(inter, "intermediate_states")
    _dev(accepted, "accepted", torch.int32)
    ss, st, sh, n_inter = _inter_strides(inter, state)
    a = make_args(None, None, None, state, slot_idx, None, None, nk=1)
    extra = (inter.data_ptr(), ss, st, sh, n_inter, accepted.data_ptr())
    return Prepared(load_library().gdr_rollback, a, extra, (state, slot_idx, inter, accepted),
                    state.device)
