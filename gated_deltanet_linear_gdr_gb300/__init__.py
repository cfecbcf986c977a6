"""GB300-native gated delta rule (GDR) recurrence.

The compute path is hand-written CUDA for sm_103a in ``csrc/``, built into the
in-tree ``libgdr.so`` behind the C ABI of ``include/gdr.h``.  This package's
Python layer is the ctypes binding over that library (marshalling only) and
the seeded synthetic workload generators.  There is no CPU fallback: the
entry points raise if the library has not been built.
"""
from ._binding import (  # noqa: F401
    GDR_BF16,
    GDR_F32,
    GdrError,
    HostForward,
    gdr_fold,
    gdr_fwd,
    gdr_fwd_conv,
    gdr_fwd_dense,
    gdr_fwd_snapshots,
    gdr_get_status,
    gdr_output_shape,
    gdr_probe_fma,
    gdr_ring_record_elements,
    gdr_rollback,
    gdr_verify_ring,
    Prepared,
    load_library,
    prepare_fold,
    prepare_fwd,
    prepare_fwd_conv,
    prepare_fwd_snapshots,
    prepare_rollback,
    prepare_verify_ring,
    status_names,
)

__version__ = "0.1.0"
