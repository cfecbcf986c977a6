"""Host-side bookkeeping of bench.py that needs no GPU: the DRAM-traffic
figure is reported only for the kernel sources it was captured on, and the
kernel-source hash ignores the host API layer but not the device code."""
from __future__ import annotations

import json
import os
import shutil

import bench


def _tree(tmp_path):
    """A copy of the kernel sources and the committed traffic summary."""
    src = os.path.join(bench.ROOT, "gated_deltanet_linear_gdr_gb300", "csrc")
    dst = tmp_path / "gated_deltanet_linear_gdr_gb300" / "csrc"
    shutil.copytree(src, dst)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, "profiles", "traffic.json"), tmp_path / "profiles")
    return dst


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash()
    path = tmp_path / "profiles" / "traffic.json"
    d = json.loads(path.read_text())
    d["k_decode_bf16_128"]["source_hash"] = h
    d["k_decode_bf16_128"]["dram_bytes_per_launch"] = 123456
    path.write_text(json.dumps(d))
    assert bench.ncu_traffic("k_decode_bf16_128") == 123456.0
    assert bench.ncu_traffic("no_such_kernel") is None

    # the host API layer checks arguments and picks kernels: not part of the hash
    with open(csrc / "api.cu", "a") as f:
        f.write("\n// host-side edit\n")
    assert bench.kernel_source_hash() == h
    assert bench.ncu_traffic("k_decode_bf16_128") == 123456.0

    # any device-side edit makes the stored counters stale
    with open(csrc / "k_decode.cu", "a") as f:
        f.write("\n// device-side edit\n")
    assert bench.kernel_source_hash() != h
    assert bench.ncu_traffic("k_decode_bf16_128") is None


def test_traffic_summary_names_every_reported_kernel():
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for key in ("k_decode_bf16_128", "k_short_verify_bf16_128", "k_fold_pair_bf16_128",
                "k_chain_snap_f32_128", "k_chain_fwd_bf16_128"):
        e = d[key]
        # each figure is rounded to whole bytes on its own
        assert abs(e["dram_bytes_per_launch"] - e["dram_bytes_read"] - e["dram_bytes_write"]) <= 2
        assert "--clock-control none" in e["command"]
        assert len(e["source_hash"]) == 16
