"""Host-side checks of the C ABI: the library builds and loads, exports every
symbol include/gdr.h declares (and nothing else), and rejects invalid
arguments before touching CUDA.  No compute call is made here."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

from gated_deltanet_linear_gdr_gb300 import _binding as B
from gated_deltanet_linear_gdr_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr.h")


@pytest.fixture(scope="module")
def lib():
    path = libbuild.build()
    return B.load_library(path)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdr_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["gdr_fwd", "gdr_fwd_conv", "gdr_verify_ring", "gdr_fold", "gdr_fwd_snapshots", "gdr_rollback",
              "gdr_output_shape", "gdr_ring_record_elements", "gdr_last_error", "gdr_get_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_library_exports_nothing_else(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    syms = {s for s in syms if not s.startswith("_") or s.startswith("gdr")}
    assert syms == set(declared_functions()), syms ^ set(declared_functions())


@pytest.mark.parametrize("cls,name", [(B.gdr_step_args, "gdr_step_args"), (B.gdr_conv_args, "gdr_conv_args")])
def test_struct_layout_matches_header(tmp_path, cls, name):
    """The ctypes mirror has the C compiler's size and field offsets for the
    struct in include/gdr.h."""
    fields = [f[0] for f in cls._fields_]
    prog = tmp_path / "layout.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gdr.h"\nint main(void) {\n'
                    f'  printf("size %zu\\n", sizeof({name}));\n' +
                    "".join(f'  printf("{f} %zu\\n", offsetof({name}, {f}));\n' for f in fields) +
                    "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                        check=True).stdout.splitlines())
    assert int(got["size"]) == ctypes.sizeof(cls)
    for f in fields:
        assert int(got[f]) == getattr(cls, f).offset, f


def test_helpers(lib):
    assert lib.gdr_version() == 100
    shp = (ctypes.c_int64 * 2)()
    assert lib.gdr_output_shape(647, 32, 128, shp) == 0
    assert (shp[0], shp[1]) == (647, 4096)
    assert lib.gdr_output_shape(-1, 32, 128, shp) == B.GDR_ERR_INVALID_ARG
    assert lib.gdr_ring_record_elements(128, 128, 2) == 392
    assert lib.gdr_ring_record_elements(16, 16, 1) == 40
    assert lib.gdr_ring_record_elements(64, 64, 5) == 64 + 8 + 320
    assert lib.gdr_ring_record_elements(0, 16, 1) == B.GDR_ERR_INVALID_ARG


def _valid_args():
    a = B.gdr_step_args()
    a.batch, a.nv, a.nk, a.K, a.V = 2, 4, 2, 16, 16
    a.state_dtype = B.GDR_BF16
    a.total_tokens = 8
    fake = 0x7f0000000000  # never dereferenced: every case below fails validation first
    a.qkv, a.qkv_seq_stride, a.qkv_chan_stride = fake, 2 * 2 * 16 + 4 * 16, 1
    a.decay, a.beta, a.tok_seq_stride, a.tok_head_stride = fake, fake, 4, 1
    a.out, a.out_seq_stride, a.out_vdim_stride = fake, 64, 1
    a.state = fake
    a.state_slot_stride, a.state_head_stride, a.state_kdim_stride, a.state_vdim_stride = (
        4 * 256, 256, 16, 1)
    a.max_slots = 4
    a.slot_idx = a.offsets = fake
    a.eps = 1e-6
    return a


BAD = [
    ("V not K, 2K or K/2", lambda a: setattr(a, "V", 48), B.GDR_ERR_UNSUPPORTED),
    ("V = K/2 at K = 16", lambda a: setattr(a, "V", 8), B.GDR_ERR_UNSUPPORTED),
    ("K unsupported", lambda a: (setattr(a, "K", 48), setattr(a, "V", 48)), B.GDR_ERR_UNSUPPORTED),
    ("nv % nk", lambda a: setattr(a, "nk", 3), B.GDR_ERR_INVALID_ARG),
    ("nv <= 0", lambda a: setattr(a, "nv", 0), B.GDR_ERR_INVALID_ARG),
    ("batch < 0", lambda a: setattr(a, "batch", -1), B.GDR_ERR_INVALID_ARG),
    ("dtype", lambda a: setattr(a, "state_dtype", 7), B.GDR_ERR_UNSUPPORTED),
    ("vdim stride", lambda a: setattr(a, "state_vdim_stride", 2), B.GDR_ERR_UNSUPPORTED),
    ("misaligned state", lambda a: setattr(a, "state", 0x7f0000000002), B.GDR_ERR_UNSUPPORTED),
    ("misaligned kdim stride", lambda a: setattr(a, "state_kdim_stride", 17), B.GDR_ERR_UNSUPPORTED),
    ("null state", lambda a: setattr(a, "state", None), B.GDR_ERR_INVALID_ARG),
    ("null slot_idx", lambda a: setattr(a, "slot_idx", None), B.GDR_ERR_INVALID_ARG),
    ("null qkv", lambda a: setattr(a, "qkv", None), B.GDR_ERR_INVALID_ARG),
    ("null out", lambda a: setattr(a, "out", None), B.GDR_ERR_INVALID_ARG),
    ("null offsets", lambda a: setattr(a, "offsets", None), B.GDR_ERR_INVALID_ARG),
    ("max_slots", lambda a: setattr(a, "max_slots", 0), B.GDR_ERR_INVALID_ARG),
    ("T < 0", lambda a: setattr(a, "total_tokens", -5), B.GDR_ERR_INVALID_ARG),
    ("zero stride", lambda a: setattr(a, "qkv_seq_stride", 0), B.GDR_ERR_INVALID_ARG),
    ("eps < 0", lambda a: setattr(a, "eps", -1.0), B.GDR_ERR_INVALID_ARG),
]


@pytest.mark.parametrize("name,mutate,code", BAD, ids=[b[0] for b in BAD])
def test_fwd_rejects_invalid_arguments(lib, name, mutate, code):
    a = _valid_args()
    mutate(a)
    assert lib.gdr_fwd(ctypes.byref(a), None) == code
    assert lib.gdr_last_error().decode()  # a message is set
    assert lib.gdr_fwd(None, None) == B.GDR_ERR_INVALID_ARG


def test_verify_and_fold_reject_bad_ring(lib):
    a = _valid_args()
    a.V = a.K = 16
    a.state = 0x7f0000000002  # still invalid: proves the ring is checked only after args...
    a.state = 0x7f0000000000
    fake = 0x7f0000000000
    need = lib.gdr_ring_record_elements(16, 16, 2)
    a.state_dtype = B.GDR_F32
    # bad ring dtype, length, stride, alignment, null pointers
    assert lib.gdr_verify_ring(ctypes.byref(a), fake, 7, 4, 8, need, fake, None) == \
        B.GDR_ERR_UNSUPPORTED
    assert need % 8 == 0
    assert lib.gdr_verify_ring(ctypes.byref(a), fake, B.GDR_BF16, 4, 8, need + 4, fake, None) == \
        B.GDR_ERR_INVALID_ARG  # a bfloat16 record stride must keep 16-byte records
    assert lib.gdr_verify_ring(ctypes.byref(a), fake + 4, B.GDR_F32, 4, 8, need, fake, None) == \
        B.GDR_ERR_UNSUPPORTED  # the verify pass writes 16-byte vectors
    assert lib.gdr_verify_ring(ctypes.byref(a), fake + 8, B.GDR_BF16, 4, 8, need, fake, None) == \
        B.GDR_ERR_UNSUPPORTED
    # the fold reads elements: an element-aligned ring passes the ring checks and
    # stops at the missing counts
    assert lib.gdr_fold(ctypes.byref(a), fake + 4, B.GDR_F32, 4, 8, need, fake, None, None) == \
        B.GDR_ERR_INVALID_ARG
    assert lib.gdr_fold(ctypes.byref(a), fake + 2, B.GDR_BF16, 4, 8, need, fake, None, None) == \
        B.GDR_ERR_INVALID_ARG
    assert lib.gdr_fold(ctypes.byref(a), fake + 2, B.GDR_F32, 4, 8, need, fake, None, None) == \
        B.GDR_ERR_UNSUPPORTED
    assert lib.gdr_verify_ring(ctypes.byref(a), fake, B.GDR_F32, 4, 0, need, fake, None) == \
        B.GDR_ERR_UNSUPPORTED
    assert lib.gdr_verify_ring(ctypes.byref(a), fake, B.GDR_F32, 4, 33, need, fake, None) == \
        B.GDR_ERR_UNSUPPORTED
    assert lib.gdr_verify_ring(ctypes.byref(a), fake, B.GDR_F32, 4, 8, need - 4, fake, None) == \
        B.GDR_ERR_INVALID_ARG
    assert lib.gdr_verify_ring(ctypes.byref(a), fake, B.GDR_F32, 4, 8, need + 2, fake, None) == \
        B.GDR_ERR_INVALID_ARG
    assert lib.gdr_verify_ring(ctypes.byref(a), None, B.GDR_F32, 4, 8, need, fake, None) == \
        B.GDR_ERR_INVALID_ARG
    assert lib.gdr_fold(ctypes.byref(a), fake, B.GDR_F32, 4, 8, need, fake, None, None) == \
        B.GDR_ERR_INVALID_ARG  # counts NULL
    assert lib.gdr_fold(ctypes.byref(a), fake, B.GDR_F32, 0, 8, need, fake, fake, None) == \
        B.GDR_ERR_INVALID_ARG  # ring_rows 0


def test_verify_and_fold_need_v_equal_k(lib):
    a = _valid_args()
    a.V = 32  # 2K: fine for the forward pass, not for the ring
    a.state_dtype = B.GDR_F32
    fake = 0x7f0000000000
    need = lib.gdr_ring_record_elements(16, 32, 2)
    assert lib.gdr_verify_ring(ctypes.byref(a), fake, B.GDR_F32, 4, 8, need, fake, None) == \
        B.GDR_ERR_UNSUPPORTED
    assert lib.gdr_fold(ctypes.byref(a), fake, B.GDR_F32, 4, 8, need, fake, fake, None) == \
        B.GDR_ERR_UNSUPPORTED
    a.K, a.V = 64, 32  # K/2: also forward-only
    need = lib.gdr_ring_record_elements(64, 32, 2)
    assert lib.gdr_verify_ring(ctypes.byref(a), fake, B.GDR_F32, 4, 8, need, fake, None) == \
        B.GDR_ERR_UNSUPPORTED
    assert lib.gdr_fold(ctypes.byref(a), fake, B.GDR_F32, 4, 8, need, fake, fake, None) == \
        B.GDR_ERR_UNSUPPORTED


def test_fwd_dense_rejects_bad_buffers(lib):
    a = _valid_args()
    a.state = a.slot_idx = None  # ignored by the dense entry point
    a.max_slots = 0
    fake = 0x7f0000000000
    assert lib.gdr_fwd_dense(ctypes.byref(a), None, None, None) == B.GDR_ERR_INVALID_ARG
    assert lib.gdr_fwd_dense(ctypes.byref(a), fake + 8, None, None) == B.GDR_ERR_UNSUPPORTED
    assert lib.gdr_fwd_dense(ctypes.byref(a), fake, fake + 8, None) == B.GDR_ERR_UNSUPPORTED
    a.V = 48  # V neither K nor 2K, as for every entry point
    assert lib.gdr_fwd_dense(ctypes.byref(a), fake, fake, None) == B.GDR_ERR_UNSUPPORTED


def test_verify_rejects_per_element_beta(lib):
    a = _valid_args()
    a.V = a.K = 16
    a.state_dtype = B.GDR_F32
    fake = 0x7f0000000000
    need = lib.gdr_ring_record_elements(16, 16, 2)
    a.beta_seq_stride, a.beta_head_stride, a.beta_vdim_stride = 64, 16, 1
    assert lib.gdr_verify_ring(ctypes.byref(a), fake, B.GDR_F32, 4, 8, need, fake, None) == \
        B.GDR_ERR_UNSUPPORTED
    a.beta_vdim_stride = -1
    assert lib.gdr_fwd(ctypes.byref(a), None) == B.GDR_ERR_INVALID_ARG


def test_snapshots_and_rollback_reject_bad_buffers(lib):
    a = _valid_args()
    fake = 0x7f0000000000
    a.state_dtype = B.GDR_F32
    hs = 16 * 16
    assert lib.gdr_fwd_snapshots(ctypes.byref(a), fake, 4 * 4 * hs, 4 * hs, hs, 4, 0, None) == \
        B.GDR_ERR_INVALID_ARG  # steps_per_token 0
    assert lib.gdr_fwd_snapshots(ctypes.byref(a), None, 4 * 4 * hs, 4 * hs, hs, 4, 2, None) == \
        B.GDR_ERR_INVALID_ARG
    assert lib.gdr_fwd_snapshots(ctypes.byref(a), fake, 4 * 4 * hs, 4 * hs, hs, 0, 2, None) == \
        B.GDR_ERR_INVALID_ARG
    assert lib.gdr_fwd_snapshots(ctypes.byref(a), fake + 4, 4 * 4 * hs, 4 * hs, hs, 4, 2, None) == \
        B.GDR_ERR_UNSUPPORTED
    assert lib.gdr_rollback(ctypes.byref(a), fake, 4 * 4 * hs, 4 * hs, hs, 4, None, None) == \
        B.GDR_ERR_INVALID_ARG
    assert lib.gdr_rollback(ctypes.byref(a), fake, 4 * 4 * hs, 4 * hs + 1, hs, 4, fake, None) == \
        B.GDR_ERR_UNSUPPORTED


def test_binding_rejects_short_intermediate_buffer():
    """The kernels index intermediate_states by pool slot, so the binding refuses
    a buffer with fewer slot rows than the pool (host-side check, no GPU)."""
    import torch
    state = torch.zeros((6, 2, 16, 16))
    with pytest.raises(ValueError, match="slot rows"):
        B._inter_strides(torch.zeros((5, 3, 2, 16, 16)), state)
    assert B._inter_strides(torch.zeros((6, 3, 2, 16, 16)), state)[3] == 3


def test_fwd_conv_rejects_bad_arguments(lib):
    a = _valid_args()
    a.state_dtype = B.GDR_F32
    fake = 0x7f0000000000
    c = B.gdr_conv_args()
    c.width, c.activation = 4, 1
    c.weight, c.weight_chan_stride, c.weight_tap_stride = fake, 4, 1
    c.conv_state = fake
    c.state_slot_stride, c.state_chan_stride, c.state_tap_stride = 96 * 3, 3, 1
    assert lib.gdr_fwd_conv(ctypes.byref(a), None, None) == B.GDR_ERR_INVALID_ARG
    for field, value, code in [("width", 0, B.GDR_ERR_UNSUPPORTED), ("width", 5, B.GDR_ERR_UNSUPPORTED),
                               ("activation", 2, B.GDR_ERR_INVALID_ARG), ("weight", None, B.GDR_ERR_INVALID_ARG),
                               ("weight_tap_stride", 0, B.GDR_ERR_INVALID_ARG),
                               ("conv_state", None, B.GDR_ERR_INVALID_ARG),
                               ("state_chan_stride", 0, B.GDR_ERR_INVALID_ARG)]:
        bad = B.gdr_conv_args.from_buffer_copy(c)
        setattr(bad, field, value)
        assert lib.gdr_fwd_conv(ctypes.byref(a), ctypes.byref(bad), None) == code, field
    # width 1 needs no conv state
    one = B.gdr_conv_args.from_buffer_copy(c)
    one.width, one.conv_state = 1, None
    a.batch = 0
    assert lib.gdr_fwd_conv(ctypes.byref(a), ctypes.byref(one), None) == B.GDR_OK
    a.batch = 2
    a.V = 32  # the fused convolution takes V = K only
    assert lib.gdr_fwd_conv(ctypes.byref(a), ctypes.byref(c), None) == B.GDR_ERR_UNSUPPORTED
    a.V = 16
    a.beta_seq_stride, a.beta_head_stride, a.beta_vdim_stride = 64, 16, 1
    assert lib.gdr_fwd_conv(ctypes.byref(a), ctypes.byref(c), None) == B.GDR_ERR_UNSUPPORTED


def test_empty_batch_is_a_no_op(lib):
    a = _valid_args()
    a.batch = 0
    assert lib.gdr_fwd(ctypes.byref(a), None) == B.GDR_OK


def test_status_null_pointer(lib):
    assert lib.gdr_get_status(None, 0) == B.GDR_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU or Python fallback"):
        B.load_library(str(tmp_path / "libgdr.so"))


def test_host_io_layout_matches_header(tmp_path):
    fields = [f[0] for f in B.gdr_host_io._fields_]
    prog = tmp_path / "hostio.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gdr.h"\nint main(void) {\n'
                    '  printf("size %zu\\n", sizeof(gdr_host_io));\n' +
                    "".join(f'  printf("{f} %zu\\n", offsetof(gdr_host_io, {f}));\n' for f in fields) +
                    "  return 0;\n}\n")
    exe = tmp_path / "hostio"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                        check=True).stdout.splitlines())
    assert int(got["size"]) == ctypes.sizeof(B.gdr_host_io)
    for f in fields:
        assert int(got[f]) == getattr(B.gdr_host_io, f).offset, f


def test_fwd_host_rejects_bad_arguments(lib):
    """Host-side checks of gdr_fwd_host, all before any CUDA call."""
    fake = 0x7f0000000000  # device pointers are never dereferenced on these paths
    off = (ctypes.c_int32 * 3)(0, 5, 8)
    io = B.gdr_host_io(fake, fake, fake, fake, ctypes.addressof(off), fake)
    call = lambda a, h: lib.gdr_fwd_host(ctypes.byref(a), h, 0, None, None, None)
    assert call(_valid_args(), None) == B.GDR_ERR_INVALID_ARG
    a = _valid_args()
    a.nk = 3  # the shared checks run first
    assert call(a, ctypes.byref(io)) == B.GDR_ERR_INVALID_ARG
    missing = B.gdr_host_io(fake, None, fake, fake, ctypes.addressof(off), fake)
    assert call(_valid_args(), ctypes.byref(missing)) == B.GDR_ERR_INVALID_ARG
    for name, value in [("qkv_seq_stride", 132), ("tok_seq_stride", 8), ("out_seq_stride", 68),
                        ("qkv_chan_stride", 2)]:
        a = _valid_args()
        setattr(a, name, value)
        assert call(a, ctypes.byref(io)) == B.GDR_ERR_UNSUPPORTED, name
    a = _valid_args()
    a.beta_seq_stride, a.beta_head_stride, a.beta_vdim_stride = 64, 16, 1
    assert call(a, ctypes.byref(io)) == B.GDR_ERR_UNSUPPORTED
    for bad in [(0, 6, 5), (0, 5, 9), (-1, 5, 8)]:
        o = (ctypes.c_int32 * 3)(*bad)
        h = B.gdr_host_io(fake, fake, fake, fake, ctypes.addressof(o), fake)
        assert call(_valid_args(), ctypes.byref(h)) == B.GDR_ERR_INVALID_ARG, bad
    a = _valid_args()
    a.batch = 0
    assert call(a, ctypes.byref(io)) == B.GDR_OK


def test_fwd_host_noalloc_rejects_bad_arguments(lib):
    """Checks of gdr_fwd_host_noalloc that come before its device set-up."""
    fake = 0x7f0000000000
    off = (ctypes.c_int32 * 3)(0, 5, 8)
    io = B.gdr_host_io(fake, fake, fake, fake, ctypes.addressof(off), fake)
    call = lambda a: lib.gdr_fwd_host_noalloc(ctypes.byref(a) if a is not None else None,
                                              ctypes.byref(io), 0, None, None, None)
    assert call(None) == B.GDR_ERR_INVALID_ARG
    a = _valid_args()
    a.nv = 0
    assert call(a) == B.GDR_ERR_INVALID_ARG
    a = _valid_args()
    a.beta_seq_stride, a.beta_head_stride, a.beta_vdim_stride = 64, 16, 1
    assert call(a) == B.GDR_ERR_UNSUPPORTED
    a = _valid_args()
    a.total_tokens = 1 << 20  # far beyond the library's staging array
    assert call(a) == B.GDR_ERR_UNSUPPORTED
    assert b"staging" in lib.gdr_last_error()



def test_probe_fma_rejects_bad_arguments(lib):
    """The diagnostic probe checks its arguments before any CUDA call."""
    n = ctypes.c_int32(0)
    fake = 0x7f0000000000
    for pattern, warps, iters, sink, ctas in [(3, 1, 1, fake, ctypes.byref(n)), (-1, 1, 1, fake, ctypes.byref(n)),
                                              (0, 0, 1, fake, ctypes.byref(n)), (0, 9, 1, fake, ctypes.byref(n)),
                                              (0, 1, 0, fake, ctypes.byref(n)), (0, 1, 1, None, ctypes.byref(n)),
                                              (0, 1, 1, fake, None)]:
        assert lib.gdr_probe_fma(pattern, warps, iters, sink, 1 << 20, ctas, None) == B.GDR_ERR_INVALID_ARG
