#!/usr/bin/env python3
"""Benchmark of the GB300 gated delta rule (GDR) recurrence.

One JSON line on stdout (rank 0).  The headline workload is the Qwen3.5-shaped
decode step: batch 256 rows x 1 token (8 padding rows), nk=16, nv=32,
K=V=128, float32 per-token inputs, bf16 state pool [512, 32, 128, 128] read
and written in place.  `value` is head-tokens/s (live tokens x nv per step /
step time) with inputs resident in HBM; `e2e` is the same metric through the
C-ABI host-buffer entry point gdr_fwd_host (binding: HostForward): the step's
inputs are copied from pinned host memory and the output copied back inside
the timed region, row groups pipelined against the compute.  The L2 cache is flushed
(a read-only sweep of a 2x-L2 buffer) before every timed step.

Secondary workloads (ragged prefill, verify + fold, Gated Delta Product
snapshots + rollback) are timed the same way and reported under "secondary".

--impl reference times the CPU oracle (oracle/, float64 C loops, one thread)
on the same decode workload and metric.

Multi-GPU (torchrun): every rank runs its own decode batch on its own GPU (the
rows of a batch are independent, so the shards exchange nothing); value is the
head-tokens of all ranks over the slowest rank's time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN recurrence head-tokens/s (decode, verify+fold); achieved HBM GB/s vs peak"
UNIT = "head-tokens/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gdr", choices=["gdr", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["prefill", "prefill_dense", "prefill_v2k", "prefill_conv", "verify_fold",
                                       "verify_fold_bf16_ring",
                                       "gdp_snapshots",
                                       "gdp_snapshots_beta_per_value"],
                    default=None,
                    help="time just this secondary workload and print its figures (profiling aid)")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="seconds of untimed steps after warm-up (steady clocks)")
    ap.add_argument("--fma-probe", action="store_true",
                    help="print the FP32-pipe rate of packed float32x2 arithmetic by register-operand pattern "
                         "(the recurrence sweep's own sequence included) and exit")
    ap.add_argument("--copy-bandwidth", action="store_true",
                    help="print the pinned host<->device copy bandwidth against copy size and exit "
                         "(the link the end-to-end figure runs over)")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers ---

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """Hash of the device code and its launchers (every csrc file but the
    host-side API layer, api.cu, which checks arguments and picks kernels)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_deltanet_linear_gdr_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")) and f != "api.cu":
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else null)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel_key]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = (uuid or "").lower().replace("gpu-", "")
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            if self.uuid and self.uuid not in f[1].lower().replace("gpu-", ""):
                continue
            try:
                rows.append((float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------- workloads ---

def decode_bytes(w, sb):
    """Algorithmic HBM bytes of one decode/forward call: each live row's state
    read and written once, each live token's q, k, v, decay, beta read and its
    output written, a padding token's zeroed output, and the index arrays."""
    conv = 2 * w.nk * w.K + w.nv * w.V
    live = w.slot_idx >= 0
    L = w.row_lengths
    live_tok = int(L[live].sum())
    pad_tok = int(L[~live].sum())
    live_rows = int(((L > 0) & live).sum())
    state = live_rows * w.nv * w.K * w.V * sb * 2
    act = live_tok * (conv + 2 * w.nv + w.nv * w.V) * 4 + pad_tok * w.nv * w.V * 4
    idx = w.batch * 4 + (w.batch + 1) * 4
    return state + act + idx


def reduce_over_ranks(local_ms: float, local_units: int, world: int, device=None):
    """Whole-job throughput across ranks: the slowest rank's time, all ranks' units.
    Returns (max_ms, total_units).  With world == 1 this is the identity."""
    if world <= 1:
        return float(local_ms), int(local_units)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    n = torch.tensor([int(local_units)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


def fma_ops(head_tokens, K, V, per=4):
    return head_tokens * per * K * V


def fp32_fma_peak(dev):
    """FMA-pipe operations per second: SMs x 128 lanes x SM clock (2.07 GHz
    when the device does not report its clock)."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    clk = getattr(props, "clock_rate", 0) * 1e3 or 2.07e9
    return props.multi_processor_count * 128 * clk


# ------------------------------------------------------------- GPU side ---

class DecodeStep:
    """Device-resident decode workload plus pinned host copies for e2e."""

    def __init__(self, w, dev):
        import numpy as np
        import torch
        self.w = w
        self.dev = dev
        self.h = {
            "qkv": torch.from_numpy(w.qkv).pin_memory(),
            "decay": torch.from_numpy(w.decay).pin_memory(),
            "beta": torch.from_numpy(w.beta).pin_memory(),
            "slot": torch.from_numpy(w.slot_idx).pin_memory(),
            "off": torch.from_numpy(w.offsets).pin_memory(),
        }
        self.d = {k: v.to(dev) for k, v in self.h.items()}
        pool = w.state_pool()
        self.state = torch.from_numpy(pool.view(np.int16)).to(dev).view(torch.bfloat16) \
            if pool.dtype == np.uint16 else torch.from_numpy(pool).to(dev)
        del pool
        self.out = torch.empty((w.total_tokens, w.nv * w.V), dtype=torch.float32, device=dev)
        self.h_out = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.h.values())
        self.d2h_bytes = self.out.numel() * 4
        import gated_deltanet_linear_gdr_gb300 as gdr
        d = self.d
        # marshalled once: the timed device path is the C-ABI call alone
        self.call = gdr.prepare_fwd(d["qkv"], d["decay"], d["beta"], self.state, d["slot"],
                                    d["off"], self.out, max_row_len=1)
        self.stream = torch.cuda.current_stream(dev).cuda_stream
        # end to end: the host-buffer entry point (tokens copied in, row groups
        # pipelined against the compute, output copied back, in one C-ABI call)
        self.host_fwd = gdr.HostForward(self.state, w.nk, w.batch, w.total_tokens, max_row_len=1)

    def run(self):
        self.call(self.stream)

    def run_e2e(self):
        h = self.h
        self.host_fwd(h["qkv"], h["decay"], h["beta"], h["slot"], h["off"], self.h_out, self.stream)


def time_steps(fn, steps, flush, stream):
    """Per-step CUDA-event durations (ms) on `stream`, L2 flushed before each."""
    import torch
    evs = []
    for _ in range(steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def _to_dev(x, dev):
    import torch
    return torch.from_numpy(x).to(dev)


def _pool_dev(w, dev):
    import numpy as np
    import torch
    pool = w.state_pool(w.live_slots())
    if pool.dtype == np.uint16:
        return torch.from_numpy(pool.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(pool).to(dev)


def bench_prefill(dev, flush, stream, hbm_peak, steps, V=0):
    """Ragged prefill (FP32-FMA bound): rows of 512..4096 tokens."""
    import torch
    import gated_deltanet_linear_gdr_gb300 as gdr
    from gated_deltanet_linear_gdr_gb300 import workloads as W
    w = W.prefill(V=V)
    st = _pool_dev(w, dev)
    qkv, dec, bet, slot, off = (_to_dev(x, dev) for x in (w.qkv, w.decay, w.beta, w.slot_idx, w.offsets))
    out = torch.empty((w.total_tokens, w.nv * w.V), device=dev)
    fn = gdr.prepare_fwd(qkv, dec, bet, st, slot, off, out)
    for _ in range(2):
        fn()
    ms = statistics.median(time_steps(fn, max(3, steps // 10), flush, stream))
    ht = w.live_head_tokens
    fp32_peak = fp32_fma_peak(dev)
    return {
        "workload": f"ragged prefill: {w.batch} rows, lengths {w.row_lengths.min()}..{w.row_lengths.max()}"
                    f" (T={w.total_tokens}), nk=16, nv=32, K={w.K}, V={w.V}, bf16 pool [16,32,{w.K},{w.V}]",
        "ms": ms, "head_tokens_per_s": ht / (ms * 1e-3),
        "fma_tflops_equiv": fma_ops(ht, w.K, w.V) / (ms * 1e-3) / 1e12,
        "fp32_fma_peak_tops": fp32_peak / 1e12,
        "frac_fp32_fma": fma_ops(ht, w.K, w.V) / (ms * 1e-3) / fp32_peak,
        "hbm_gbs": decode_bytes(w, 2) / (ms * 1e-3) / 1e9,
    }


def bench_prefill_conv(dev, flush, stream, hbm_peak, steps):
    """The ragged prefill workload from the RAW Pass-1 input: the causal
    depthwise convolution (width 4, SiLU, bias) fused into the recurrence's
    operand staging, then the conv-state update (gdr_fwd_conv)."""
    import torch
    import gated_deltanet_linear_gdr_gb300 as gdr
    from gated_deltanet_linear_gdr_gb300 import workloads as W
    w = W.prefill()
    cv = W.conv_inputs(w, width=4, seed=2)
    st = _pool_dev(w, dev)
    x, dec, bet, slot, off = (_to_dev(a, dev) for a in (w.qkv, w.decay, w.beta, w.slot_idx, w.offsets))
    wt, bs, cs = (_to_dev(a, dev) for a in (cv.weight, cv.bias, cv.state))
    out = torch.empty((w.total_tokens, w.nv * w.V), device=dev)
    fn = gdr.prepare_fwd_conv(x, dec, bet, st, slot, off, wt, bs, cs, out)
    for _ in range(2):
        fn()
    ms = statistics.median(time_steps(fn, max(3, steps // 10), flush, stream))
    ht = w.live_head_tokens
    fp32_peak = fp32_fma_peak(dev)
    return {
        "workload": f"ragged prefill from the raw Pass-1 input: {w.batch} rows, T={w.total_tokens}, nk=16, nv=32, "
                    "K=V=128, bf16 pool [16,32,128,128], conv width 4 + bias + SiLU fused, conv state "
                    "[16,8192,3] fp32",
        "ms": ms, "head_tokens_per_s": ht / (ms * 1e-3),
        "frac_fp32_fma": fma_ops(ht, w.K, w.V) / (ms * 1e-3) / fp32_peak,
    }


def bench_prefill_v2k(dev, flush, stream, hbm_peak, steps):
    """The ragged prefill workload with value heads twice the key heads (V = 256)."""
    return bench_prefill(dev, flush, stream, hbm_peak, steps, V=256)


def bench_prefill_dense(dev, flush, stream, hbm_peak, steps):
    """The ragged prefill workload with a dense start and end state
    (initial_state given, final state written to a second tensor)."""
    import numpy as np
    import torch
    import gated_deltanet_linear_gdr_gb300 as gdr
    from gated_deltanet_linear_gdr_gb300 import workloads as W
    w = W.prefill()
    pool = w.state_pool(w.live_slots())
    init = torch.from_numpy(pool[w.slot_idx].view(np.int16)).to(dev).view(torch.bfloat16)
    final = torch.empty_like(init)
    qkv, dec, bet, off = (_to_dev(x, dev) for x in (w.qkv, w.decay, w.beta, w.offsets))
    out = torch.empty((w.total_tokens, w.nv * w.V), device=dev)
    a = gdr._binding.make_args(qkv, dec, bet, init, torch.zeros(w.batch, dtype=torch.int32, device=dev),
                               off, out, nk=w.nk)
    fn_c = gdr.load_library().gdr_fwd_dense
    import ctypes

    def fn():
        gdr._binding._check(fn_c(ctypes.byref(a), init.data_ptr(), final.data_ptr(), stream.cuda_stream))
    for _ in range(2):
        fn()
    ms = statistics.median(time_steps(fn, max(3, steps // 10), flush, stream))
    ht = w.live_head_tokens
    return {
        "workload": f"ragged prefill, dense state: {w.batch} rows, T={w.total_tokens}, bf16 initial/final "
                    f"[{w.batch},32,128,128]",
        "ms": ms, "head_tokens_per_s": ht / (ms * 1e-3),
        "frac_fp32_fma": fma_ops(ht, w.K, w.V) / (ms * 1e-3) / fp32_fma_peak(dev),
    }


def bench_verify_fold(dev, flush, stream, hbm_peak, steps, ring_dtype=None):
    """Speculative verify (bf16 pool, fp32 or bf16 ring of RING_LEN 8) then fold."""
    import torch
    import gated_deltanet_linear_gdr_gb300 as gdr
    from gated_deltanet_linear_gdr_gb300 import workloads as W
    w = W.verify_fold()
    st = _pool_dev(w, dev)
    qkv, dec, bet, slot, off = (_to_dev(x, dev) for x in (w.qkv, w.decay, w.beta, w.slot_idx, w.offsets))
    ring_dtype = ring_dtype or torch.float32
    stride = (gdr.gdr_ring_record_elements(w.K, w.V, w.nv // w.nk) + 7) // 8 * 8
    ring = torch.zeros((w.ring_rows, w.nk, w.ring_len, stride), dtype=ring_dtype, device=dev)
    rb = ring.element_size()
    rsi, cnt = _to_dev(w.ring_slot_idx, dev), _to_dev(w.counts, dev)
    out = torch.empty((w.total_tokens, w.nv * w.V), device=dev)
    # the caller of a verify window knows its longest row: the short-row kernel
    v_fn = gdr.prepare_verify_ring(qkv, dec, bet, st, slot, off, ring, rsi, out,
                                   max_row_len=int(w.row_lengths.max()))
    f_fn = gdr.prepare_fold(st, slot, ring, rsi, cnt)
    for _ in range(2):
        v_fn()
        f_fn()
    tv = statistics.median(time_steps(v_fn, steps, flush, stream))
    tf = statistics.median(time_steps(f_fn, steps, flush, stream))
    L = w.row_lengths
    short = L <= w.ring_len
    r = w.nv // w.nk
    rec = w.K + ((r + 7) // 8) * 8 + r * w.V
    conv = 2 * w.nk * w.K + w.nv * w.V
    vbytes = (w.batch * w.nv * w.K * w.V * 2 + int((~short).sum()) * w.nv * w.K * w.V * 2
              + w.total_tokens * (conv + 2 * w.nv + w.nv * w.V) * 4
              + int(L[short].sum()) * w.nk * rec * rb)
    active = (w.counts > 0) & (w.counts <= w.ring_len) & (w.slot_idx >= 0)
    fbytes = (int(active.sum()) * w.nv * w.K * w.V * 2 * 2
              + int(w.counts[active].sum()) * w.nk * rec * rb)
    ht = w.live_head_tokens
    # roofline time of each kernel: the larger of its HBM time and its FMA-pipe time
    fp32_peak = fp32_fma_peak(dev)
    v_roof = max(vbytes / (hbm_peak * 1e9), fma_ops(ht, w.K, w.V) / fp32_peak)
    f_roof = max(fbytes / (hbm_peak * 1e9),
                 fma_ops(int(w.counts[active].sum()) * w.nv, w.K, w.V, per=2) / fp32_peak)
    return {
        "workload": "verify: 127 rows x 5 drafts + 1 row of 12, RING_LEN 8, nk=16, nv=32, "
                    f"K=V=128, bf16 pool [256,32,128,128], "
                    f"{'bf16' if rb == 2 else 'fp32'} ring [256,16,8,{stride}]; then fold "
                    "of accepted counts ~U{0..5}",
        "verify_ms": tv, "fold_ms": tf, "head_tokens_per_s": ht / ((tv + tf) * 1e-3),
        "verify_hbm_gbs": vbytes / (tv * 1e-3) / 1e9, "fold_hbm_gbs": fbytes / (tf * 1e-3) / 1e9,
        "frac_hbm_verify_plus_fold": (vbytes + fbytes) / ((tv + tf) * 1e-3) / 1e9 / hbm_peak,
        "roofline_us_verify": v_roof * 1e6, "roofline_us_fold": f_roof * 1e6,
        "frac_roofline_verify_plus_fold": (v_roof + f_roof) / ((tv + tf) * 1e-3),
    }


def bench_gdp_snapshots(dev, flush, stream, hbm_peak, steps, beta_per_value=False):
    """Gated Delta Product drafts with snapshots (fp32 cache), then rollback."""
    import torch
    import gated_deltanet_linear_gdr_gb300 as gdr
    from gated_deltanet_linear_gdr_gb300 import workloads as W
    w = W.gdp_snapshots(beta_per_value=beta_per_value)
    st = _pool_dev(w, dev)
    qkv, dec, bet, slot, off = (_to_dev(x, dev) for x in (w.qkv, w.decay, w.beta, w.slot_idx, w.offsets))
    inter = torch.zeros((w.max_slots, w.n_inter, w.nv, w.K, w.V), device=dev)
    acc = _to_dev(w.accepted, dev)
    out = torch.empty((w.total_tokens, w.nv * w.V), device=dev)
    s_fn = gdr.prepare_fwd_snapshots(qkv, dec, bet, st, slot, off, inter, w.steps_per_token, out,
                                     decay_is_log=True, max_row_len=int(w.row_lengths.max()))
    r_fn = gdr.prepare_rollback(st, slot, inter, acc)
    for _ in range(2):
        s_fn()
        r_fn()
    ts = statistics.median(time_steps(s_fn, steps, flush, stream))
    tr = statistics.median(time_steps(r_fn, steps, flush, stream))
    sbytes = decode_bytes(w, 4) + w.batch * w.n_inter * w.nv * w.K * w.V * 4
    if beta_per_value:  # beta [T, nv, V] instead of [T, nv]
        sbytes += w.total_tokens * w.nv * (w.V - 1) * 4
    rbytes = w.batch * w.nv * w.K * w.V * 4 * 2
    ht = w.live_head_tokens
    return {
        "workload": "GDP spec-decode: 64 requests x 4 drafts x 2 Householder copies (T=8 each), "
                    "spt=2, nk=16, nv=32, K=V=128, fp32 cache [128,32,128,128], "
                    "intermediate [128,4,32,128,128]"
                    + (", beta per value element [T,32,128]" if beta_per_value else "")
                    + "; then rollback",
        "snapshots_ms": ts, "rollback_ms": tr, "head_tokens_per_s": ht / (ts * 1e-3),
        "snapshots_hbm_gbs": sbytes / (ts * 1e-3) / 1e9, "rollback_hbm_gbs": rbytes / (tr * 1e-3) / 1e9,
        "frac_hbm_snapshots": sbytes / (ts * 1e-3) / 1e9 / hbm_peak,
        "frac_hbm_rollback": rbytes / (tr * 1e-3) / 1e9 / hbm_peak,
    }


def bench_verify_fold_bf16_ring(dev, flush, stream, hbm_peak, steps):
    """The verify + fold workload with a bfloat16 ring (records rounded once)."""
    import torch
    return bench_verify_fold(dev, flush, stream, hbm_peak, steps, ring_dtype=torch.bfloat16)


def bench_gdp_snapshots_beta_per_value(dev, flush, stream, hbm_peak, steps):
    """The snapshot workload with beta per value element (general kernel)."""
    return bench_gdp_snapshots(dev, flush, stream, hbm_peak, steps, beta_per_value=True)


SECONDARY = {"prefill": bench_prefill, "prefill_dense": bench_prefill_dense, "prefill_v2k": bench_prefill_v2k,
             "prefill_conv": bench_prefill_conv,
             "verify_fold": bench_verify_fold,
             "verify_fold_bf16_ring": bench_verify_fold_bf16_ring,
             "gdp_snapshots": bench_gdp_snapshots,
             "gdp_snapshots_beta_per_value": bench_gdp_snapshots_beta_per_value}


def secondary(dev, flush, stream, hbm_peak, steps, only=None):
    """The non-headline workloads, each timed like decode (L2 flushed per step)."""
    import torch
    res = {}
    for name, fn in SECONDARY.items():
        if only is None or only == name:
            res[name] = fn(dev, flush, stream, hbm_peak, steps)
            torch.cuda.empty_cache()
    return res


# ---------------------------------------------------- CPU baseline (oracle) ---
# The oracle (float64 C loops, test infrastructure) timed on the host's cores
# as it stands: rows and key-head groups are independent, so a workload is cut
# into independent pieces and the pieces are run on Python threads (the C
# oracle runs with the GIL released).  Single-thread and all-core figures.

def host_cpu():
    """(logical CPUs, CPU model string) of the host the oracle runs on."""
    n = os.cpu_count() or 1
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip().lower() in ("model name", "cpu model", "hardware") and v.strip():
                    model = v.strip()
                    break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                k, _, v = line.partition(":")
                if k.strip() in ("Model name", "Vendor ID") and v.strip():
                    model = (model + " " + v.strip()).strip()
        except (OSError, subprocess.SubprocessError):
            pass
    import platform
    return n, f"{model or 'unknown'} ({platform.machine()})"


def cpu_piece(w, rows, heads=None, t_max=None):
    """An independent piece of workload w as oracle.Problem arguments: rows
    `rows` (each cut to its first t_max tokens), key heads `heads` (all when
    None) with their value heads, and a compact pool holding only those rows'
    slots (padding rows keep slot -1)."""
    import numpy as np
    nk, K, V = w.nk, w.K, w.V
    r = w.nv // nk
    hks = list(range(nk)) if heads is None else list(heads)
    vh = [hk * r + j for hk in hks for j in range(r)]
    toks, offs, slots, states = [], [0], [], []
    for i, b in enumerate(rows):
        t0, t1 = int(w.offsets[b]), int(w.offsets[b + 1])
        if t_max is not None:
            t1 = min(t1, t0 + t_max)
        toks.extend(range(t0, t1))
        offs.append(offs[-1] + t1 - t0)
        live = int(w.slot_idx[b]) >= 0
        slots.append(i if live else -1)
        states.append(w.state_slot(int(w.slot_idx[b]))[vh] if live else None)
    dt = np.uint16 if w.state_dtype == "bf16" else np.float32
    pool = np.zeros((len(rows), len(vh), K, V), dt)
    for i, st in enumerate(states):
        if st is not None:
            pool[i] = st
    toks = np.asarray(toks, dtype=np.int64)
    cols = ([c for hk in hks for c in range(hk * K, (hk + 1) * K)]
            + [nk * K + c for hk in hks for c in range(hk * K, (hk + 1) * K)]
            + [2 * nk * K + h * V + j for h in vh for j in range(V)])
    beta = w.beta[toks][:, vh] if w.beta.ndim == 2 else w.beta[toks][:, vh, :]
    return dict(qkv=w.qkv[toks][:, cols], decay=w.decay[toks][:, vh], beta=beta, state=pool,
                slot_idx=np.asarray(slots, np.int32), offsets=np.asarray(offs, np.int32),
                nk=len(hks), nv=len(vh), K=K, V=V, decay_is_log=w.decay_is_log,
                use_l2norm=w.use_l2norm, scale=w.scale, eps=w.eps)


def _cpu_time(pieces, run_piece, threads):
    """Wall seconds to run every piece once on `threads` threads."""
    from concurrent.futures import ThreadPoolExecutor
    t0 = time.perf_counter()
    if threads <= 1:
        for pc in pieces:
            run_piece(pc)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(run_piece, pieces))
    return time.perf_counter() - t0


def cpu_baseline(kind, w, budget_s=4.0, t_max=None):
    """The oracle on workload w (kind: "fwd", "verify_fold", "snapshots"):
    head-tokens/s on one thread and on every host core.  The sample is the
    whole workload, or each row's first t_max tokens."""
    import numpy as np
    import oracle
    ncpu, model = host_cpu()
    L = np.diff(w.offsets.astype(np.int64))
    if t_max is not None:
        L = np.minimum(L, t_max)
    head_tokens = int(L[w.slot_idx >= 0].sum()) * w.nv
    rows = list(range(w.batch))
    # pieces: one row (with every head) for short rows, one (row, key head) for long ones
    by_head = t_max is not None or w.total_tokens > 4 * w.batch
    pieces = []
    for b in rows:
        for hk in (range(w.nk) if by_head else [None]):
            pc = cpu_piece(w, [b], None if hk is None else [hk], t_max)
            if w.counts is not None:
                pc["counts"] = w.counts[[b]].astype(np.int32)
            if w.accepted is not None:
                pc["accepted"] = w.accepted[[b]].astype(np.int32)
            pieces.append(pc)
    r = w.nv // w.nk

    def run_piece(pc):
        args = {k: v for k, v in pc.items() if k not in ("counts", "accepted")}
        args["state"] = args["state"].copy()
        prob = oracle.Problem(**args)
        if kind == "fwd":
            oracle.fwd(prob)
        elif kind == "verify_fold":
            nb = len(args["slot_idx"])
            rec = oracle.ring_record_elements(prob.K, prob.V, r)
            ring = np.zeros((nb, prob.nk, w.ring_len, rec), np.float32)
            rsi = np.arange(nb, dtype=np.int32)
            oracle.verify_ring(prob, ring, rsi, w.ring_len)
            oracle.fold(prob, ring, rsi, pc["counts"], w.ring_len)
        else:
            nb = prob.state.shape[0]
            inter = np.zeros((nb, w.n_inter, prob.nv, prob.K, prob.V), prob.state.dtype)
            oracle.fwd_snapshots(prob, inter, w.steps_per_token)
            oracle.rollback(prob, inter, pc["accepted"])

    res = {}
    for threads in (1, ncpu):
        rounds, secs = 0, 0.0
        while secs < budget_s and rounds < 50:
            secs += _cpu_time(pieces, run_piece, threads)
            rounds += 1
        res[threads] = (head_tokens * rounds / secs, rounds, secs)
    all_v, all_r, all_s = res[ncpu]
    one_v, one_r, one_s = res[1]
    sample = (f"{'first ' + str(t_max) + ' tokens of each row' if t_max else 'the whole workload'} "
              f"({head_tokens} live head-tokens per round), float64 C loops; rows"
              f"{' and key heads' if by_head else ''} run as {len(pieces)} independent "
              f"pieces on {ncpu} threads: {all_r} rounds in {all_s:.1f} s; one thread: {one_r} rounds in "
              f"{one_s:.1f} s")
    return {"value": all_v, "unit": UNIT, "cores": ncpu, "kind": "oracle", "sample": sample,
            "single_thread": {"value": one_v, "unit": UNIT, "cores": 1},
            "host": {"nproc": ncpu, "cpu": model}}


def _cpu_workloads():
    """Secondary workloads that get a CPU baseline: (oracle pass, workload, tokens per row sampled)."""
    from gated_deltanet_linear_gdr_gb300 import workloads as W
    return {
        # the prefill sample: each row's first 256 tokens (the whole rows take minutes)
        "prefill": ("fwd", W.prefill, 256),
        "verify_fold": ("verify_fold", W.verify_fold, None),
        "gdp_snapshots": ("snapshots", W.gdp_snapshots, None),
    }


def cpu_baseline_decode(w, budget_s=5.0):
    """The CPU oracle on whole decode batches, one thread and every host core."""
    return cpu_baseline("fwd", w, budget_s)


def run_gdr(args):
    import numpy as np
    import torch
    import torch.distributed as dist
    import gated_deltanet_linear_gdr_gb300 as gdr
    from gated_deltanet_linear_gdr_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    gdr.load_library()
    stream = torch.cuda.current_stream(dev)

    if args.only:
        props = torch.cuda.get_device_properties(dev)
        flush_buf = torch.zeros(max(2 * getattr(props, "L2_cache_size", 128 << 20), 256 << 20) // 4,
                                dtype=torch.float32, device=dev)
        res = secondary(dev, lambda: flush_buf.sum(), stream, peaks()[0], args.steps, only=args.only)
        print(json.dumps({"only": args.only, **res.get(args.only, {})}), flush=True)
        return
    w = W.decode(seed=1 + rank)
    step = DecodeStep(w, dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20)
    flush_buf = torch.zeros(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)

    def flush():
        # read-only sweep of 2x L2: evicts our lines without leaving dirty ones behind
        flush_buf.sum()

    hbm_peak, peak_kind = peaks()
    uuid = str(getattr(props, "uuid", "")) or None
    sampler = ClockSampler(uuid)

    for _ in range(max(3, args.warmup)):
        flush()
        step.run()
    torch.cuda.synchronize()
    sampler.start()
    t_end = time.time() + args.soak_s
    while time.time() < t_end:
        for _ in range(20):
            flush()
            step.run()
        torch.cuda.synchronize()

    # ---- timed region: exactly `steps` steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    per = time_steps(step.run, args.steps, flush, stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    st = gdr.gdr_get_status(clear=True)
    if st:
        raise RuntimeError(f"device status after timed region: {gdr.status_names(st)}")

    ht = w.live_head_tokens
    kernel_ms_max, units = reduce_over_ranks(sum(per), ht * args.steps, world, dev)
    ms_per_step = kernel_ms_max / args.steps
    value = units / (kernel_ms_max * 1e-3)

    # ---- end-to-end through the public API with host buffers
    for _ in range(3):
        step.run_e2e()
    torch.cuda.synchronize()
    per_e2e = time_steps(step.run_e2e, args.steps, flush, stream)
    e2e_ms, e2e_units = reduce_over_ranks(sum(per_e2e), ht * args.steps, world, dev)
    e2e_value = e2e_units / (e2e_ms * 1e-3)

    alg_bytes = decode_bytes(w, 2)
    achieved = alg_bytes / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": DECODE_WORKLOAD,
            "global_batch": 256 * world, "seq_len": 1, "parallelism": f"dp{world}",
            "l2": "flushed before every timed step (read-only sweep of a 2x-L2 buffer)",
            "head_tokens_per_step": ht * world,
            "alg_bytes_per_step": alg_bytes,
            "timed_wall_s": wall,
        },
        "roofline": {
            "bound": "hbm", "kernel": "gdr::k_decode_pipe<bf16,128,3>", "achieved": achieved,
            "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
            "peak_kind": f"{peak_kind} (STREAM-style copy)",
            "traffic": ncu_traffic("k_decode_bf16_128"),
        },
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": step.h2d_bytes,
                "d2h_bytes_per_step": step.d2h_bytes},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_secondary:
        try:
            line["secondary"] = secondary(dev, flush, stream, hbm_peak, max(5, args.steps // 2))
        except Exception as e:  # report, never hide
            line["secondary"] = {"error": repr(e)}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(w)
        sec = line.get("secondary")
        if isinstance(sec, dict) and "error" not in sec:
            for name, (kind, wl, t_max) in _cpu_workloads().items():
                if name in sec:
                    sec[name]["cpu_baseline"] = cpu_baseline(kind, wl(), t_max=t_max)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# The headline workload, named the same way by both arms.
DECODE_WORKLOAD = ("decode: batch 256 rows x 1 token (248 live, 8 padding slot -1), nk=16, nv=32, K=V=128, "
                   "fp32 q/k/v/decay/beta, bf16 state pool [512,32,128,128] at random slots")


def run_reference(args):
    """The CPU oracle as it stands, on the decode workload, on every host core
    (rank 0 only): each step runs the whole decode batch as independent rows
    on one thread per core."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from gated_deltanet_linear_gdr_gb300 import workloads as W
    w = W.decode()
    ncpu, model = host_cpu()
    pieces = [cpu_piece(w, [b]) for b in range(w.batch)]

    def run_piece(pc):
        args_ = dict(pc)
        args_["state"] = args_["state"].copy()
        oracle.fwd(oracle.Problem(**args_))

    for _ in range(max(1, args.warmup)):
        _cpu_time(pieces, run_piece, ncpu)
    times = [_cpu_time(pieces, run_piece, ncpu) for _ in range(args.steps)]
    total = sum(times)
    ht = w.live_head_tokens
    value = ht * args.steps / total
    sample = (f"whole decode batch per step (256 rows, {ht} live head-tokens), float64 C loops, rows as "
              f"independent pieces on {ncpu} threads")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": DECODE_WORKLOAD, "global_batch": 256, "seq_len": 1, "parallelism": "dp1",
                   "runs_on": "host cores (the CPU oracle)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": ncpu, "kind": "oracle", "sample": sample,
                         "host": {"nproc": ncpu, "cpu": model}},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def copy_bandwidth(steps=20):
    """Pinned host<->device copy bandwidth against copy size: one cudaMemcpyAsync
    per copy on its own stream, CUDA events around it, median of `steps`; also
    both directions at once on two streams (the overlap gdr_fwd_host uses)."""
    import torch
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    rows = []
    decode_in = DECODE_H2D_BYTES
    sizes = sorted({64 << 10, 256 << 10, 1 << 20, 4 << 20, decode_in, 16 << 20, 64 << 20, 256 << 20})
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    for n in sizes:
        h_in = torch.empty(n // 4, dtype=torch.float32).pin_memory()
        h_out = torch.empty(n // 4, dtype=torch.float32).pin_memory()
        d_a = torch.empty(n // 4, dtype=torch.float32, device=dev)
        d_b = torch.empty(n // 4, dtype=torch.float32, device=dev)

        def timed(fn, stream):
            ts = []
            for _ in range(steps + 3):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                b.synchronize()
                ts.append(a.elapsed_time(b))
            return statistics.median(ts[3:]) * 1e-3

        with torch.cuda.stream(s1):
            t_h2d = timed(lambda: d_a.copy_(h_in, non_blocking=True), s1)
            t_d2h = timed(lambda: h_out.copy_(d_b, non_blocking=True), s1)

        def both():
            e = torch.cuda.Event()
            e.record(s1)
            s2.wait_event(e)
            with torch.cuda.stream(s1):
                d_a.copy_(h_in, non_blocking=True)
            with torch.cuda.stream(s2):
                h_out.copy_(d_b, non_blocking=True)
            f = torch.cuda.Event()
            f.record(s2)
            s1.wait_event(f)
        t_both = timed(both, s1)
        rows.append({"bytes": n, "h2d_gbs": n / t_h2d / 1e9, "d2h_gbs": n / t_d2h / 1e9,
                     "h2d_us": t_h2d * 1e6, "d2h_us": t_d2h * 1e6,
                     "both_directions_gbs": 2 * n / t_both / 1e9})
    print(json.dumps({"copy_bandwidth": rows, "pinned": True,
                      "method": "one cudaMemcpyAsync per copy, CUDA events on its stream, median of "
                                f"{steps}"}), flush=True)


def fma_probe(steps=7):
    """FP32-pipe rate of packed float32x2 arithmetic with every operand in
    registers, by operand pattern and warps per SM sub-partition (gdr_probe_fma):
    the ceiling the recurrence kernels' fixed operation order can reach on the
    FMA pipe.  CUDA events on the launching stream, median of `steps`, the SM
    clock sampled during the runs."""
    import torch
    from gated_deltanet_linear_gdr_gb300 import GdrError, gdr_probe_fma
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    sink = torch.empty(sms * 128 * 8, dtype=torch.float32, device=dev)
    # FP32 operations per thread per iteration, and iterations per launch
    ops = {0: 512, 1: 16, 2: 16}
    iters = {0: 1024, 1: 16384, 2: 16384}
    names = {0: "recurrence sweep (t = alpha x; x = k u + t; a += x k; b += x q), 64 rows x 2 columns",
             1: "packed FMA chains, multiplier and addend shared by every instruction",
             2: "packed FMA chains, three distinct operand registers per instruction"}
    clocks = ClockSampler(str(getattr(props, "uuid", "")))
    clocks.start()
    rows = []
    for pattern in (1, 2, 0):
        for w in (1, 2, 4, 8):
            try:
                gdr_probe_fma(pattern, w, iters[pattern], sink)
            except GdrError:
                continue  # the pattern's CTA does not fit one SM at this warp count
            ts = []
            for _ in range(steps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                ctas = gdr_probe_fma(pattern, w, iters[pattern], sink)
                b.record(stream)
                b.synchronize()
                ts.append(a.elapsed_time(b) * 1e-3)
            t = statistics.median(ts)
            n = ctas * 128 * w * iters[pattern] * ops[pattern]
            rows.append({"pattern": pattern, "what": names[pattern], "warps_per_subpartition": w,
                         "us": t * 1e6, "fp32_ops_per_s": n / t})
    clk = clocks.stop()
    mhz = clk.get("sm_mhz") or 2070.0
    for r in rows:
        r["ops_per_sm_per_cycle"] = r["fp32_ops_per_s"] / sms / (mhz * 1e6)
        r["frac_of_fp32_peak"] = r["ops_per_sm_per_cycle"] / 128
    print(json.dumps({"fma_probe": rows, "clocks": clk, "sms": sms,
                      "peak": "128 FP32 lane operations per SM per cycle (an FMA or a multiply counts "
                              "as one, as in the roofline's FMA-pipe count)"}), flush=True)


# Pinned host bytes one decode step copies in (q/k/v, decay, beta, slot_idx, offsets).
DECODE_H2D_BYTES = 256 * (2 * 16 * 128 + 32 * 128) * 4 + 2 * 256 * 32 * 4 + 256 * 4 + 257 * 4


def main():
    args = parse()
    if args.copy_bandwidth:
        copy_bandwidth()
        return
    if args.fma_probe:
        fma_probe()
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gdr(args)


if __name__ == "__main__":
    main()
