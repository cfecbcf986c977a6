"""gdr_fwd_host_noalloc: the host-buffer forward pass for callers that cannot
allocate device memory (for instance a plug-in handed only host buffers and a
stream, or code inside a stream capture that forbids allocation).  It stages
the tokens in the library's own fixed device array instead of buffers from the
caller; its results must equal gdr_fwd_host's (same kernels, same order of
operations: bit for bit), call after call, since every call reuses the array.

Kept in a file of its own, collected last, so that a run stopping at the
first failure has already run every other test."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import gated_deltanet_linear_gdr_gb300 as gdr
import gated_deltanet_linear_gdr_gb300._binding as B
from gated_deltanet_linear_gdr_gb300 import workloads as W
from tests.gpu_helpers import DEV, pool_to_dev, pool_to_host

pytestmark = pytest.mark.gpu


def _pinned(x):
    return torch.from_numpy(np.ascontiguousarray(x)).pin_memory()


@pytest.mark.parametrize("case", ["decode", "ragged"])
def test_no_alloc_entry_point_matches_host_forward_twice(case):
    if case == "decode":
        w = W.decode(batch=64, max_slots=96, n_pad=2)
        mrl = 1
    else:
        w = W.random_case(97, [6, 0, 11, 3, 8], nk=2, nv=4, K=64, max_slots=8, state_dtype="bf16",
                          n_pad=1)
        mrl = 0
    gdr.gdr_get_status(clear=True)
    pool = w.state_pool()
    lib = gdr.load_library()
    stream = torch.cuda.current_stream(DEV).cuda_stream
    host = [_pinned(x) for x in (w.qkv, w.decay, w.beta, w.slot_idx, w.offsets)]
    shape = (w.total_tokens, w.nv * w.V)

    # the existing entry point, with device buffers of the caller's
    ref_state = pool_to_dev(pool)
    hf = gdr.HostForward(ref_state, w.nk, w.batch, w.total_tokens, decay_is_log=w.decay_is_log,
                         use_qk_l2norm=w.use_l2norm, scale=w.scale, eps=w.eps, max_row_len=mrl)
    # the no-alloc entry point: the same arguments, its own staging array
    state = pool_to_dev(pool)
    args = B.gdr_step_args.from_buffer_copy(hf.args)
    args.state = state.data_ptr()

    for call in range(2):  # the pool advances in place: two steps in a row
        ref_out = torch.full(shape, float("nan")).pin_memory()
        hf(*host, ref_out)
        out = torch.full(shape, float("nan")).pin_memory()
        io = B.gdr_host_io(*(t.data_ptr() for t in host), out.data_ptr())
        rc = lib.gdr_fwd_host_noalloc(ctypes.byref(args), ctypes.byref(io), 0, stream,
                                      hf.h2d.cuda_stream, hf.d2h.cuda_stream)
        assert rc == 0, lib.gdr_last_error()
        torch.cuda.synchronize()
        assert (out.numpy().view(np.uint32) == ref_out.numpy().view(np.uint32)).all(), call
        assert (pool_to_host(state) == pool_to_host(ref_state)).all(), call
    assert gdr.gdr_get_status() == 0


def test_no_alloc_entry_point_rejects_calls_beyond_its_array():
    """A call whose staging would not fit the fixed array is refused before
    anything is copied or launched, with a message saying why."""
    w = W.random_case(98, [4, 4], nk=2, nv=4, K=64, max_slots=4, state_dtype="bf16")
    state = pool_to_dev(w.state_pool())
    lib = gdr.load_library()
    hf = gdr.HostForward(state, w.nk, w.batch, w.total_tokens)
    args = B.gdr_step_args.from_buffer_copy(hf.args)
    args.total_tokens = 1 << 20  # 1M tokens x 2 KiB of qkv each: far beyond the array
    io = B.gdr_host_io(1, 1, 1, 1, 1, 1)  # never touched: the size check comes first
    before = pool_to_host(state)
    rc = lib.gdr_fwd_host_noalloc(ctypes.byref(args), ctypes.byref(io), 0,
                                  torch.cuda.current_stream(DEV).cuda_stream, None, None)
    assert rc == B.GDR_ERR_UNSUPPORTED
    assert b"staging" in lib.gdr_last_error()
    torch.cuda.synchronize()
    assert (pool_to_host(state) == before).all()
