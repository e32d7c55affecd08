#!/usr/bin/env python3
"""Benchmark of the block-scaled quantization hot path on one GB300 per rank.

One step = one pass of the hot path over the NVFP4 dense workload
(BF16 M=8192 x K=7168, N(0,1) x per-row LogNormal(0,1) with 0.1% x50
outliers, tensor_sf = 448*6/global amax): ``bsq_quantize`` (packed E2M1 +
E4M3 scales in the 5D TCGEN layout) and ``bsq_scales_interleave`` of the
rank-2 form of the result's scales.  The two are independent, so the
reinterleave runs on a second stream: it is forked from the main stream at
the start of each step (after the previous step's quantize) and both streams
are joined once, before the closing event of the timed region.  The serial
form (both on one stream) is reported beside it.  The metric is GB/s over the
algorithmic bytes (BF16 in + packed out + scale bytes; 2 bytes per scale for
the reinterleave), with the inputs resident in HBM.  Steps cycle through
three copies of every buffer (352 MB of BF16 input, larger than the 129 MB
L2), so no step finds its data in L2.  Kernels are timed with CUDA events on
the stream they are launched on.

Also reported on the same JSON line: ``e2e`` (the same metric through the
Python API with pinned host buffers, host<->device copies inside the timed
region), ``roofline`` for the dominant kernel (dense quantize), ``clocks``
sampled with nvidia-smi during the timed region, ``cpu_baseline`` (the CPU
oracle on a bounded sample, rank 0 at N=1) and ``workloads`` (the other
shapes: NVFP4 128x256, MXFP8/MXFP4 16384x4096, grouped prefill with the
top-8 gather and with the rows already permuted (32768 and 8192 rows),
grouped decode in
microseconds per k_tiles_per_block, the tensor scales and the chains).

``--impl reference`` times the CPU oracle itself on the same workload, one
bounded sample per step.

Multi-GPU: launched under torchrun, every rank quantizes its own batch of the
same shape on its own GPU (weak scaling, no collective on the data path); the
step time is the max over ranks and ``value`` counts the bytes of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "quantize GB/s (bytes in+out) and % of GB300 HBM peak; grouped decode µs"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
ROTATE = 3
CSRC = os.path.join(ROOT, "fp8_activation_quantization_bsq_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dense_nvfp4_M8192_K7168.traffic.json")
REF_SAMPLE_ROWS = 256
CPU_BASELINE_ROWS = 8192


# ----------------------------------------------------------------- helpers --

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def bf16_peak():
    """Dense bf16 TFLOP/s (burst) from MEASURED_PEAKS.json, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback 1900 TFLOP/s"


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


DENSE_SOURCES = ("device_common.cuh", "box_quant.cuh", "dense_quant.cuh")


def source_digest() -> str:
    """sha256 over the dense kernel's source files (the profiled kernel)."""
    h = hashlib.sha256()
    for name in DENSE_SOURCES:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def profiled_traffic():
    """DRAM bytes per launch of the dense kernel from the committed ncu summary,
    or None when missing or taken on different kernel sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("source_sha256") != source_digest():
        return None
    return t.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples, kept only inside a window."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [r for (t, r) in self.rows if t0 <= t <= t1 + 0.06]
        note = "samples inside the timed region"
        if not inside and self.rows:
            # the region was shorter than the sampling period: take the nearest sample
            inside = [min(self.rows, key=lambda tr: abs(tr[0] - (t0 + t1) / 2))[1]]
            note = "timed region shorter than the 50 ms sampling period: nearest sample"
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            try:
                sm.append(float(r[2]))
                smax.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "note": note}


def to_dev_bf16(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def rank2_from_5d(scales5d, M, S):
    """Torch view of a 5D scale buffer as (M, S) row-major bytes (setup only)."""
    Mt, Kt = -(-M // 128), -(-S // 4)
    v = scales5d[: Mt * Kt * 512].view(Mt, Kt, 32, 4, 4).permute(0, 3, 2, 1, 4)
    return v.reshape(Mt * 128, Kt * 4)[:M, :S].contiguous()


def dense_bytes(fmt: str, M: int, K: int) -> int:
    sf = 16 if fmt == "nvfp4" else 32
    out = M * (K if fmt == "mxfp8" else K // 2)
    return M * K * 2 + out + M * (K // sf)


# --------------------------------------------------------------- GPU timing --

def gpu_hold(ms: float) -> None:
    """Queue a bounded spin kernel of about ``ms`` milliseconds, outside any
    timed events, so that the host has enqueued the work that follows before
    the device reaches it: timed launches then run back to back, with no gaps
    from host-side enqueue cost inside the events."""
    import torch
    torch.cuda._sleep(int(ms * 1e-3 * 2.0e9))


def time_events(fn, reps: int, flush=None, prep=None):
    """Mean / min device ms of fn() over reps, CUDA events on the current
    stream.  With ``flush`` (a buffer of 2x the L2 size) a read pass over it
    runs before each rep, outside the events: it evicts earlier data and
    writes back dirty lines, leaving L2 clean (cold-cache timing).  ``prep``
    (enqueued before the flush) reads what a consumer of the previous rep's
    outputs would read."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    torch.cuda.synchronize()
    gpu_hold(1.0 + 0.15 * reps)
    for i, (a, b) in enumerate(evs):
        if prep is not None:
            prep()
        if flush is not None:
            flush.sum(dtype=torch.int32)
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    return statistics.mean(ms), min(ms)


E2E_SLABS = 4       # row slabs of one end-to-end step (copies overlapped with the kernels)
ROT_SETS = 3        # buffer sets cycled by the back-to-back context timings
ROT_LAUNCHES = 30


class ScaleList(list):
    """A list of launch closures that also keeps their scale buffers."""
    def __init__(self):
        super().__init__()
        self.scales = []


def time_rotated(fns, launches: int = ROT_LAUNCHES):
    """Device ms per launch of ``launches`` launches back to back, cycling
    through ``fns`` (one per buffer set, each set larger than the L2 or the
    other sets together larger than it, so that every launch finds its own
    buffers evicted): one CUDA-event pair on the current stream around all of
    them, after one untimed launch per set."""
    import torch
    for f in fns:
        f()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_hold(1.0 + 0.06 * launches)
    a.record()
    for i in range(launches):
        fns[i % len(fns)]()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / launches


def extra_workloads(bsq, device, flush, peak):
    """The other shapes, reported for context (not the headline).

    ``us``: device time per launch, launches back to back over ROT_SETS
    rotated buffer sets (inputs and outputs; cold in L2 for each launch).
    ``us_single_cold``: one launch between two events after an L2 flush,
    which adds the launch latency the back-to-back timing hides (about
    4-5 us on this GPU for a one-block kernel)."""
    import torch
    import workloads as wl
    res = {}
    reps = 30

    c = wl.config_dense_nvfp4_small()
    x = to_dev_bf16(c["x_bits"], device)
    out, sc = bsq.quantize(x, "nvfp4", float(c["tensor_sf"]))
    mean, mn = time_events(lambda: bsq.quantize(x, "nvfp4", float(c["tensor_sf"]), out=out, scales=sc), reps, flush)
    res["nvfp4_dense_M128_K256"] = {"us_single_cold": round(mean * 1e3, 2), "us_min": round(mn * 1e3, 2),
                                    "GB_s": round(dense_bytes("nvfp4", 128, 256) / (mean * 1e6), 1),
                                    "note": "one 128-row tile: launch latency"}

    # tensor-scale reduction and the on-device NVFP4 chain (tensor_sf, then
    # quantize reading it from device memory) on the 8192 x 7168 activations
    c = wl.config_dense_nvfp4_large()
    x0 = to_dev_bf16(c["x_bits"], device)
    M, K = c["x_bits"].shape
    del c
    xs = [x0] + [x0.clone() for _ in range(ROT_SETS - 1)]
    ws = torch.zeros(bsq.lib().bsq_tensor_sf_workspace_bytes(), dtype=torch.uint8, device=device)
    tsfs = [bsq.tensor_sf(x, workspace=ws) for x in xs]
    fns = [lambda x=x, t=t: bsq.tensor_sf(x, out=t, workspace=ws) for x, t in zip(xs, tsfs)]
    rot = time_rotated(fns)
    single, _ = time_events(fns[0], reps, flush)
    res[f"tensor_sf_M{M}_K{K}"] = {"us": round(rot * 1e3, 2), "GB_s": round(M * K * 2 / (rot * 1e6), 1),
                                   "frac_of_hbm": round(M * K * 2 / (rot * 1e6) / peak, 3),
                                   "us_single_cold": round(single * 1e3, 2)}
    outs = [bsq.quantize_dynamic(x, "nvfp4", t[1:]) for x, t in zip(xs, tsfs)]

    def chain(i):
        bsq.tensor_sf(xs[i], out=tsfs[i], workspace=ws)
        bsq.quantize_dynamic(xs[i], "nvfp4", tsfs[i][1:], out=outs[i][0], scales=outs[i][1])
    rot = time_rotated([lambda i=i: chain(i) for i in range(ROT_SETS)])
    single, _ = time_events(lambda: chain(0), reps, flush)
    res[f"nvfp4_dynamic_chain_M{M}_K{K}"] = {
        "us": round(rot * 1e3, 2), "us_single_cold": round(single * 1e3, 2),
        "note": "tensor_sf + quantize_dynamic; the input is read twice",
        "GB_s_of_quantize_bytes": round(dense_bytes("nvfp4", M, K) / (rot * 1e6), 1)}
    del outs, tsfs
    x = xs[0]
    del xs

    # the naive block-scaled matmul validator (FP64 CUDA cores), NVFP4
    # 512 x 512 x 7168 from the first rows of the dense workload
    xa, xb = x[:512], x[512:1024]
    pa, sa = bsq.quantize(xa, "nvfp4", 1.0)
    pb, sb = bsq.quantize(xb, "nvfp4", 1.0)
    cd = bsq.block_scaled_dot("nvfp4", pa, sa, pb, sb, K)
    mean, _ = time_events(lambda: bsq.block_scaled_dot("nvfp4", pa, sa, pb, sb, K, out=cd), 5)
    res["block_scaled_dot_nvfp4_512x512x7168"] = {"us": round(mean * 1e3, 1),
                                                  "GFLOP_s_fp64": round(2 * 512 * 512 * K / (mean * 1e6), 1)}
    del pa, sa, pb, sb, cd

    # the quantize fused into a matmul epilogue: C (8192 x 2048) = x (8192 x
    # 7168) times 2048 rows of x as the weight, NVFP4, against the separate
    # quantize of the same BF16 C
    wgt = x[4096:6144]
    cb = torch.empty((M, 2048), dtype=torch.bfloat16, device=device)
    gq, gs = bsq.gemm_quantize(x, wgt, "nvfp4", 1.0, c_out=cb)
    mean, _ = time_events(lambda: bsq.gemm_quantize(x, wgt, "nvfp4", 1.0, out=gq, scales=gs), 5, flush)
    qa, qs = bsq.quantize(cb, "nvfp4", 1.0)
    qmean, _ = time_events(lambda: bsq.quantize(cb, "nvfp4", 1.0, out=qa, scales=qs), reps, flush)
    tflops = 2 * M * 2048 * K / (mean * 1e9)
    res["nvfp4_gemm_quantize_epilogue_8192x2048x7168"] = {
        "us": round(mean * 1e3, 1), "TFLOP_s_bf16": round(tflops, 1),
        "frac_of_bf16_peak": round(tflops / bf16_peak()[0], 3), "bf16_peak_source": bf16_peak()[1],
        "separate_quantize_of_C_us_single_cold": round(qmean * 1e3, 2),
        "note": "tcgen05 mainloop (TMA operands, TMEM accumulators); the epilogue replaces a BF16 C store plus a "
                "quantize pass; one launch between events after an L2 flush"}
    del gq, gs, qa, qs, cb, wgt, x

    c = wl.config_dense_mx_wide()
    x0 = to_dev_bf16(c["x_bits"], device)
    del c
    xs = [x0] + [x0.clone() for _ in range(ROT_SETS - 1)]
    for fmt in ("mxfp8", "mxfp4"):
        outs = [bsq.quantize(x, fmt) for x in xs]
        fns = [lambda x=x, o=o: bsq.quantize(x, fmt, out=o[0], scales=o[1]) for x, o in zip(xs, outs)]
        rot = time_rotated(fns)
        single, _ = time_events(fns[0], reps, flush)
        b = dense_bytes(fmt, 16384, 4096)
        res[f"{fmt}_dense_M16384_K4096"] = {"GB_s": round(b / (rot * 1e6), 1), "us": round(rot * 1e3, 2),
                                            "frac_of_hbm": round(b / (rot * 1e6) / peak, 3),
                                            "us_single_cold": round(single * 1e3, 2)}
        del outs, fns
    del xs, x0

    def consume(tensors):
        # read the outputs once, as their consumer would: the grouped token
        # and band kernels store scale bytes with an L2 evict_last hint, and
        # an ordinary read returns those lines to normal priority, so that a
        # workload's unread scales do not stay favoured in L2 through the
        # workloads measured after it
        for t in tensors:
            t.max()
        torch.cuda.synchronize()

    def grouped_sets(d, fmt, kt, sets, workspace=False):
        """Launch closures over `sets` buffer sets (token-matrix copy, packed
        output, 5D scales, optionally the scale-staging workspace; the
        metadata shared) and the algorithmic bytes; the sets' scale buffers
        are kept in fns.scales."""
        x0 = to_dev_bf16(d["x_bits"], device)
        xgs = [x0] + [x0.clone() for _ in range(sets - 1)]
        u32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.uint32).view(np.int32)).to(device)
        ro, so = u32(d["row_offsets"]), u32(d["scales_offsets"])
        eid = torch.from_numpy(d["expert_ids"]).to(device)
        sf = torch.from_numpy(d["sf_tensor"]).to(device) if fmt == "nvfp4" else None
        ridx = torch.from_numpy(d["row_indices"]).to(device) if d["row_indices"] is not None else None
        kw = dict(total_rows=d["total_rows"], total_scale_rows=d["total_scale_rows"], k_tiles_per_block=kt)
        fns = ScaleList()
        for xg in xgs:
            out, sc = bsq.grouped_quantize(xg, fmt, ro, so, eid, sf, ridx, **kw)
            fns.scales.append(sc)
            ws = torch.empty(bsq.grouped_quantize_workspace_bytes(fmt, d["total_scale_rows"], d["K"]),
                             dtype=torch.uint8, device=device) if workspace else None
            fns.append(lambda xg=xg, out=out, sc=sc, ws=ws: bsq.grouped_quantize(
                xg, fmt, ro, so, eid, sf, ridx, out=out, scales=sc, workspace=ws, **kw))
        K = d["K"]
        sfv = 16 if fmt == "nvfp4" else 32
        kt_cols = -(-(K // sfv) // 4) * 4
        gather = d["row_indices"] is not None
        uniq = int(np.unique(d["row_indices"]).size) if gather else d["total_rows"]
        b = (uniq * K * 2 + d["total_rows"] * (K if fmt == "mxfp8" else K // 2)
             + d["total_rows"] * kt_cols + (d["row_indices"].nbytes if gather else 0) + d["row_offsets"].nbytes
             + d["scales_offsets"].nbytes + d["expert_ids"].nbytes
             + (d["sf_tensor"].nbytes if fmt == "nvfp4" else 0))
        return fns, b

    d = wl.config_grouped_prefill()
    x0 = to_dev_bf16(d["x_bits"], device)
    xgs = [x0] + [x0.clone() for _ in range(ROT_SETS - 1)]
    ro = torch.from_numpy(np.ascontiguousarray(d["row_offsets"], np.uint32).view(np.int32)).to(device)
    eid = torch.from_numpy(d["expert_ids"]).to(device)
    ridx = torch.from_numpy(d["row_indices"]).to(device)
    E = d["num_experts"]
    gws = torch.zeros(bsq.lib().bsq_grouped_tensor_sf_workspace_bytes(E), dtype=torch.uint8, device=device)
    gsfs = [bsq.grouped_tensor_sf(xg, ro, eid, E, ridx, total_rows=d["total_rows"], workspace=gws) for xg in xgs]
    fns = [lambda xg=xg, g=g: bsq.grouped_tensor_sf(xg, ro, eid, E, ridx, total_rows=d["total_rows"], out=g,
                                                    workspace=gws) for xg, g in zip(xgs, gsfs)]
    rot = time_rotated(fns)
    single, _ = time_events(fns[0], reps, flush)
    res["grouped_tensor_sf_prefill_T4096_K7168"] = {
        "us": round(rot * 1e3, 2), "us_single_cold": round(single * 1e3, 2),
        "gathered_GB_s": round(d["total_rows"] * d["K"] * 2 / (rot * 1e6), 1)}
    # the grouped dynamic chain: per-expert scales on the GPU, then the
    # grouped NVFP4 quantize reading them from device memory
    so_d = torch.from_numpy(np.ascontiguousarray(d["scales_offsets"], np.uint32).view(np.int32)).to(device)
    gkw = dict(total_rows=d["total_rows"], total_scale_rows=d["total_scale_rows"], k_tiles_per_block=8)
    gouts = [bsq.grouped_quantize(xg, "nvfp4", ro, so_d, eid, g, ridx, **gkw) for xg, g in zip(xgs, gsfs)]

    def gchain(i):
        bsq.grouped_tensor_sf(xgs[i], ro, eid, E, ridx, total_rows=d["total_rows"], out=gsfs[i], workspace=gws)
        bsq.grouped_quantize(xgs[i], "nvfp4", ro, so_d, eid, gsfs[i], ridx, out=gouts[i][0], scales=gouts[i][1],
                             **gkw)
    rot = time_rotated([lambda i=i: gchain(i) for i in range(ROT_SETS)])
    single, _ = time_events(lambda: gchain(0), reps, flush, prep=lambda: gouts[0][1].max())
    res["nvfp4_grouped_dynamic_chain_prefill_T4096_K7168"] = {"us": round(rot * 1e3, 2),
                                                             "us_single_cold": round(single * 1e3, 2)}
    # the same chain with the quantize's scale-staging workspace
    gwss = [torch.empty(bsq.grouped_quantize_workspace_bytes("nvfp4", d["total_scale_rows"], d["K"]),
                        dtype=torch.uint8, device=device) for _ in range(ROT_SETS)]

    def gchain_ws(i):
        bsq.grouped_tensor_sf(xgs[i], ro, eid, E, ridx, total_rows=d["total_rows"], out=gsfs[i], workspace=gws)
        bsq.grouped_quantize(xgs[i], "nvfp4", ro, so_d, eid, gsfs[i], ridx, out=gouts[i][0], scales=gouts[i][1],
                             workspace=gwss[i], **gkw)
    rot = time_rotated([lambda i=i: gchain_ws(i) for i in range(ROT_SETS)])
    res["nvfp4_grouped_dynamic_chain_prefill_T4096_K7168_workspace"] = {"us": round(rot * 1e3, 2)}
    del gwss
    consume([g[1] for g in gouts])
    del gouts, so_d, xgs, x0, gsfs, gws, fns
    for fmt, ws in (("nvfp4", False), ("nvfp4", True), ("mxfp8", False), ("mxfp4", False)):
        fns, b = grouped_sets(d, fmt, 8, ROT_SETS, workspace=ws)
        rot = time_rotated(fns)
        single, _ = time_events(fns[0], reps, flush, prep=lambda: fns.scales[0].max())
        res[f"{fmt}_grouped_prefill_T4096_K7168" + ("_workspace" if ws else "")] = {
            "GB_s": round(b / (rot * 1e6), 1), "us": round(rot * 1e3, 2),
            "frac_of_hbm": round(b / (rot * 1e6) / peak, 3), "us_single_cold": round(single * 1e3, 2),
            "algorithmic_bytes": b, "logical_input_bytes": d["total_rows"] * d["K"] * 2,
            "T_elements_per_s": round(d["total_rows"] * d["K"] / (rot * 1e-3) / 1e12, 2)}
        consume(fns.scales)
        del fns
    # the same groups with the rows already permuted (row_indices NULL: the
    # 32768 x 7168 input is read once, row by row)
    dn = dict(d, x_bits=d["x_bits"][d["row_indices"]], row_indices=None)
    for fmt in ("nvfp4", "mxfp8", "mxfp4"):
        fns, b = grouped_sets(dn, fmt, 8, ROT_SETS)
        rot = time_rotated(fns)
        single, _ = time_events(fns[0], reps, flush, prep=lambda: fns.scales[0].max())
        res[f"{fmt}_grouped_prefill_nogather_R32768_K7168"] = {
            "GB_s": round(b / (rot * 1e6), 1), "us": round(rot * 1e3, 2),
            "frac_of_hbm": round(b / (rot * 1e6) / peak, 3), "us_single_cold": round(single * 1e3, 2),
            "algorithmic_bytes": b, "note": "rows already permuted by expert (no row_indices)"}
        consume(fns.scales)
        del fns
    del d, dn
    # fewer rows without a gather (1024 tokens, top-8 of 256 experts, rows
    # permuted): the streaming kernel splits its column runs to fill the GPU
    d = wl.config_grouped_prefill(seed=11, tokens=1024, K=7168)
    dn = dict(d, x_bits=d["x_bits"][d["row_indices"]], row_indices=None)
    for fmt in ("nvfp4", "mxfp8", "mxfp4"):
        fns, b = grouped_sets(dn, fmt, 8, ROT_SETS)
        rot = time_rotated(fns)
        single, _ = time_events(fns[0], reps, flush, prep=lambda: fns.scales[0].max())
        res[f"{fmt}_grouped_nogather_R8192_K7168"] = {
            "GB_s": round(b / (rot * 1e6), 1), "us": round(rot * 1e3, 2),
            "frac_of_hbm": round(b / (rot * 1e6) / peak, 3), "us_single_cold": round(single * 1e3, 2),
            "algorithmic_bytes": b, "note": "1024 tokens top-8, rows already permuted (no row_indices)"}
        consume(fns.scales)
        del fns
    del d, dn
    for fmt in ("nvfp4", "mxfp8"):
        for K in (7168, 2048):
            d = wl.config_grouped_decode(K=K, fmt=fmt)
            for kt in (0, 1, 2, 4, 8):  # 0: chosen by the library
                fns, b = grouped_sets(d, fmt, kt, 1)
                mean, mn = time_events(fns[0], reps, flush, prep=lambda: fns.scales[0].max())
                warm = time_events(fns[0], reps)[0]
                b2b = time_rotated(fns)
                res[f"{fmt}_grouped_decode_T64_K{K}_kt{'auto' if kt == 0 else kt}"] = {
                    "us_single_cold": round(mean * 1e3, 2), "us_min": round(mn * 1e3, 2),
                    "us_single_warm_l2": round(warm * 1e3, 2), "us_back_to_back_warm_l2": round(b2b * 1e3, 2)}
                consume(fns.scales)
                del fns
    return res


def run_ours(args, rank, world, local_rank):
    import torch
    import fp8_activation_quantization_bsq_gb300 as bsq
    import workloads as wl

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    device = torch.device("cuda", torch.cuda.current_device() if world == 1 else local_rank)
    torch.cuda.set_device(device)
    bsq.lib()

    c = wl.config_dense_nvfp4_large(seed=1 + rank)
    M, K, tsf = c["M"], c["K"], float(c["tensor_sf"])
    S = K // 16
    x0 = to_dev_bf16(c["x_bits"], device)
    bufs = []
    for r in range(ROTATE):
        x = x0 if r == 0 else x0.clone()
        out = torch.empty((M, K // 2), dtype=torch.uint8, device=device)
        sc = torch.empty(bsq.scales5d_bytes("nvfp4", M, K), dtype=torch.uint8, device=device)
        bsq.quantize(x, "nvfp4", tsf, out=out, scales=sc)
        torch.cuda.synchronize()
        sc2d = rank2_from_5d(sc, M, S)                   # rank-2 copy of the result's scales
        bufs.append((x, out, sc, sc2d, torch.empty_like(sc)))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    side = torch.cuda.Stream(device)       # the reinterleave of each step
    fork = torch.cuda.Event()

    q_bytes = dense_bytes("nvfp4", M, K)
    il_bytes = 2 * M * S
    step_bytes = q_bytes + il_bytes

    def step(i):
        x, out, sc, sc2d, sc5 = bufs[i % ROTATE]         # data of this step is not in L2
        fork.record(stream)
        side.wait_event(fork)
        bsq.quantize(x, "nvfp4", tsf, out=out, scales=sc)
        with torch.cuda.stream(side):
            bsq.scales_interleave(sc2d, out=sc5)

    def step_serial(i):
        x, out, sc, sc2d, sc5 = bufs[i % ROTATE]
        bsq.quantize(x, "nvfp4", tsf, out=out, scales=sc)
        bsq.scales_interleave(sc2d, out=sc5)

    def join():
        stream.wait_stream(side)

    def quantize_only(i):
        x, out, sc, _, _ = bufs[i % ROTATE]
        bsq.quantize(x, "nvfp4", tsf, out=out, scales=sc)

    ev = lambda: torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # host enqueue cost of one step, to size the hold that keeps the device fed
    th = time.perf_counter()
    for i in range(5):
        step(i)
    host_ms = (time.perf_counter() - th) / 5 * 1e3
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps, CUDA events at its two ends (the
    # quantize kernels run back to back on the main stream, programmatic
    # dependent launch overlapping each launch with the previous kernel's
    # tail; the reinterleaves run beside them on the side stream, which is
    # joined before the closing event)
    sampler = ClockSampler(device.index) if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    e0, e1 = ev(), ev()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    gpu_hold(1.0 + 1.5 * host_ms * args.steps)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    join()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    clocks = sampler.stop(t0, t1) if sampler else None
    step_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    value = step_bytes * world / (step_ms * 1e-3) / 1e9

    # the same K steps with both kernels on one stream (context)
    s0, s1 = ev(), ev()
    torch.cuda.synchronize()
    gpu_hold(1.0 + 1.5 * host_ms * args.steps)
    s0.record(stream)
    for i in range(args.steps):
        step_serial(i)
    s1.record(stream)
    torch.cuda.synchronize()
    serial_ms = max_over_ranks(s0.elapsed_time(s1) / args.steps, world)

    # ---- the dominant kernel alone: K back-to-back quantize launches on the
    # same rotating buffers, events at the ends -> mean duration per launch
    q0, q1 = ev(), ev()
    torch.cuda.synchronize()
    gpu_hold(1.0 + 1.5 * host_ms * args.steps)
    q0.record(stream)
    for i in range(args.steps):
        quantize_only(i)
    q1.record(stream)
    torch.cuda.synchronize()
    q_mean = max_over_ranks(q0.elapsed_time(q1) / args.steps, world)

    # ---- end to end through the public API with pinned host buffers
    x, out, sc, sc2d, sc5 = bufs[0]
    x_h = torch.from_numpy(np.ascontiguousarray(c["x_bits"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    sc2d_h = sc2d.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=torch.uint8).pin_memory()
    sc_h = torch.empty(sc.shape, dtype=torch.uint8).pin_memory()
    sc5_h = torch.empty(sc5.shape, dtype=torch.uint8).pin_memory()
    sc2d_d = torch.empty_like(sc2d)
    h2d = x_h.numel() * 2 + sc2d_h.numel()
    d2h = out_h.numel() + sc_h.numel() + sc5_h.numel()

    def e2e_step(a, b, i):
        a.record(stream)
        x.copy_(x_h, non_blocking=True)
        sc2d_d.copy_(sc2d_h, non_blocking=True)
        bsq.quantize(x, "nvfp4", tsf, out=out, scales=sc)
        bsq.scales_interleave(sc2d_d, out=sc5)
        out_h.copy_(out, non_blocking=True)
        sc_h.copy_(sc, non_blocking=True)
        sc5_h.copy_(sc5, non_blocking=True)
        b.record(stream)

    for i in range(min(args.warmup, 3)):
        e2e_step(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True), i)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 50))
    ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    barrier(world)
    gpu_hold(2.0)
    for i, (a, b) in enumerate(ee):
        e2e_step(a, b, i)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ee), world)
    ref_out = (out_h.clone(), sc_h.clone(), sc5_h.clone())

    # the same steps pipelined: each step in E2E_SLABS row slabs (whole
    # 128-row bands), the host->device copy of a slab, its quantize +
    # reinterleave and the device->host copy of its results on three
    # streams, so copies in both directions overlap the kernels and each
    # other; a slab's device buffers are reused once its previous results
    # are back on the host
    nsl = E2E_SLABS
    rows = M // nsl
    bands = rows // 128
    s_h2d, s_d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    c_done = [torch.cuda.Event() for _ in range(nsl)]
    d_done = [torch.cuda.Event() for _ in range(nsl)]
    sc_slab = bsq.scales5d_bytes("nvfp4", rows, K)
    assert sc_slab * nsl == sc.numel() and rows % 128 == 0

    def e2e_pipelined(n_steps):
        for _ in range(n_steps):
            for k in range(nsl):
                r0, r1 = k * rows, (k + 1) * rows
                s0, s1 = k * sc_slab, (k + 1) * sc_slab
                h_done = torch.cuda.Event()
                with torch.cuda.stream(s_h2d):
                    s_h2d.wait_event(c_done[k])           # the slab's previous kernels have read it
                    x[r0:r1].copy_(x_h[r0:r1], non_blocking=True)
                    sc2d_d[r0:r1].copy_(sc2d_h[r0:r1], non_blocking=True)
                    h_done.record(s_h2d)
                stream.wait_event(h_done)
                stream.wait_event(d_done[k])              # its previous results are back on the host
                bsq.quantize(x[r0:r1], "nvfp4", tsf, out=out[r0:r1], scales=sc[s0:s1])
                bsq.scales_interleave(sc2d_d[r0:r1], out=sc5[s0:s1])
                c_done[k].record(stream)
                with torch.cuda.stream(s_d2h):
                    s_d2h.wait_event(c_done[k])
                    out_h[r0:r1].copy_(out[r0:r1], non_blocking=True)
                    sc_h[s0:s1].copy_(sc[s0:s1], non_blocking=True)
                    sc5_h[s0:s1].copy_(sc5[s0:s1], non_blocking=True)
                    d_done[k].record(s_d2h)

    e2e_pipelined(2)
    torch.cuda.synchronize()
    assert all(torch.equal(u, v) for u, v in zip(ref_out, (out_h, sc_h, sc5_h))), "pipelined e2e results differ"
    th = time.perf_counter()
    e2e_pipelined(2)
    host_e2e_ms = (time.perf_counter() - th) / 2 * 1e3   # host enqueue cost of one pipelined step
    torch.cuda.synchronize()
    barrier(world)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    gpu_hold(2.0 + 1.5 * host_e2e_ms * e2e_steps)          # the host enqueues ahead of the device
    p0.record(stream)
    s_h2d.wait_event(p0)
    s_d2h.wait_event(p0)
    e2e_pipelined(e2e_steps)
    s_d2h.wait_stream(stream)
    s_d2h.wait_stream(s_h2d)
    p1.record(s_d2h)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(p0.elapsed_time(p1) / e2e_steps, world)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    peak, peak_src = hbm_peak()
    achieved = q_bytes / (q_mean * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded NumPy PCG64; no dataset)",
        "config": {"workload": "nvfp4_dense_quantize_M8192_K7168+scales_interleave",
                   "format": "nvfp4", "M": M, "K": K, "tensor_sf": tsf,
                   "bytes_per_step": step_bytes, "quantize_bytes": q_bytes, "interleave_bytes": il_bytes,
                   "l2": "inputs larger than L2: steps cycle through 3 copies of all buffers (352 MB BF16 input)",
                   "parallelism": f"replicas x{world} (each rank its own batch)"},
        "hbm_frac": round(value / world / peak, 4),
        "streams": "quantize on the main stream, reinterleave on a side stream forked each step, joined before the closing event",
        "serial": {"ms_per_step": round(serial_ms, 5),
                   "value": round(step_bytes * world / (serial_ms * 1e-3) / 1e9, 2),
                   "note": "both kernels on one stream"},
        "e2e": {"value": round(step_bytes * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "pipelining": f"{E2E_SLABS} row slabs per step; H2D, kernels and D2H on three streams",
                "serial_value": round(step_bytes * world / (e2e_serial_ms * 1e-3) / 1e9, 2)},
        "roofline": {"bound": "hbm", "kernel": "dense_quant_tma_kernel<NVFP4>",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6800 GB/s", "us_per_launch": round(q_mean * 1e3, 3)},
        "gpu_launches": 2 * args.steps,
        "timing": "events at the two ends of the K-step region; per-launch kernel time from K back-to-back launches of the kernel alone",
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(c, tsf)
    if not args.no_extra:
        line["workloads"] = extra_workloads(bsq, device, flush, peak)
        line["workloads_timing"] = (f"us: device time per launch, {ROT_LAUNCHES} launches back to back cycling "
                                    f"through {ROT_SETS} buffer sets (inputs and outputs; each launch's own "
                                    "buffers evicted from L2 by the other sets); us_single_cold: one launch "
                                    "between events after a 2x-L2 read pass (adds the launch latency)")
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------- CPU oracle --

def oracle_sample_step(c, tsf, rows):
    """One pass of the CPU oracle over ``rows`` rows of the workload:
    quantize (rank-2 scales + 5D) and reinterleave; returns the bytes done."""
    import oracle
    bits = c["x_bits"][:rows]
    packed, s2 = oracle.quantize_rank2("nvfp4", bits, tsf)
    oracle.scales_to_5d(s2)
    oracle.scales_interleave(s2, rows, s2.shape[1], s2.shape[1])
    return dense_bytes("nvfp4", rows, c["K"]) + 2 * rows * (c["K"] // 16)


def _oracle_chunk(job):
    """Process-pool task: one 512-row chunk of the oracle step (bytes done)."""
    bits, K, tsf = job
    return oracle_sample_step({"x_bits": bits, "K": K}, tsf, bits.shape[0])


def cpu_baseline(c, tsf):
    """The oracle on the host cores: all rows of the workload in 512-row
    chunks, once on one core and once spread over a spawned process pool with
    one worker per core (spawned, because this runs after CUDA has started)."""
    chunks = [c["x_bits"][r0:r0 + 512] for r0 in range(0, CPU_BASELINE_ROWS, 512)]
    t0 = time.perf_counter()
    done = sum(_oracle_chunk((b, c["K"], tsf)) for b in chunks)
    dt1 = time.perf_counter() - t0
    one = done / dt1 / 1e9
    cores = max(1, min(os.cpu_count() or 1, len(chunks)))
    try:
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        with ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")) as pool:
            list(pool.map(_oracle_chunk, [(chunks[0][:16], c["K"], tsf)] * cores))  # workers up
            t0 = time.perf_counter()
            done_n = sum(pool.map(_oracle_chunk, [(b, c["K"], tsf) for b in chunks]))
            dtn = time.perf_counter() - t0
        many = done_n / dtn / 1e9
    except Exception as e:  # no process pool on this host: report the one-core figure
        return {"value": round(one, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"all {CPU_BASELINE_ROWS} rows in 512-row chunks, quantize + 5D + interleave, "
                          f"NumPy, one core; {dt1:.2f} s (process pool unavailable: {type(e).__name__})"}
    return {"value": round(many, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "single_core_value": round(one, 5),
            "sample": f"all {CPU_BASELINE_ROWS} rows of the workload in 512-row chunks, quantize + 5D + "
                      f"interleave, NumPy: {dt1:.2f} s on one core, {dtn:.2f} s over {cores} worker "
                      f"processes"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import workloads as wl
    c = wl.config_dense_nvfp4_large()
    tsf = np.float32(c["tensor_sf"])
    for _ in range(args.warmup):
        oracle_sample_step(c, tsf, REF_SAMPLE_ROWS)
    times, done = [], 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        done = oracle_sample_step(c, tsf, REF_SAMPLE_ROWS)
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    value = done / (ms * 1e-3) / 1e9
    sample = f"first {REF_SAMPLE_ROWS} of 8192 rows per step (quantize + 5D + interleave), NumPy single-threaded"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded NumPy PCG64; no dataset)",
            "config": {"workload": "nvfp4_dense_quantize_M8192_K7168+scales_interleave",
                       "format": "nvfp4", "M": 8192, "K": 7168, "sample_rows": REF_SAMPLE_ROWS},
            "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


CASES = ("grouped_prefill", "grouped_nogather", "grouped_decode", "tensor_sf", "grouped_tensor_sf", "mxfp8", "mxfp4",
         "gemm_quantize")


def run_case(args):
    """One context workload alone (for profiling a single kernel): warm-up
    launches, then ``--steps`` launches back to back on one GPU; prints one
    JSON line with the mean microseconds per launch (CUDA events)."""
    import torch
    import fp8_activation_quantization_bsq_gb300 as bsq
    import workloads as wl
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    if args.case in ("grouped_prefill", "grouped_nogather", "grouped_decode", "grouped_tensor_sf"):
        d = wl.config_grouped_prefill() if args.case != "grouped_decode" else wl.config_grouped_decode()
        if args.case == "grouped_nogather":  # the same groups with the rows already permuted
            d = dict(d, x_bits=d["x_bits"][d["row_indices"]], row_indices=None)
        x = to_dev_bf16(d["x_bits"], device)
        u32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.uint32).view(np.int32)).to(device)
        ro, so = u32(d["row_offsets"]), u32(d["scales_offsets"])
        eid = torch.from_numpy(d["expert_ids"]).to(device)
        sf = torch.from_numpy(d["sf_tensor"]).to(device)
        ridx = torch.from_numpy(d["row_indices"]).to(device) if d["row_indices"] is not None else None
        kw = dict(total_rows=d["total_rows"], total_scale_rows=d["total_scale_rows"], k_tiles_per_block=8)
        if args.case == "grouped_tensor_sf":
            ws = torch.zeros(bsq.lib().bsq_grouped_tensor_sf_workspace_bytes(d["num_experts"]),
                             dtype=torch.uint8, device=device)
            out = bsq.grouped_tensor_sf(x, ro, eid, d["num_experts"], ridx, total_rows=d["total_rows"],
                                        workspace=ws)
            fn = lambda: bsq.grouped_tensor_sf(x, ro, eid, d["num_experts"], ridx, total_rows=d["total_rows"],
                                               out=out, workspace=ws)
        else:
            kw["kernel"] = args.grouped_kernel
            if args.grouped_workspace:
                kw["workspace"] = torch.empty(bsq.grouped_quantize_workspace_bytes(args.fmt, d["total_scale_rows"],
                                                                                   d["K"]),
                                              dtype=torch.uint8, device=device)
            out, sc = bsq.grouped_quantize(x, args.fmt, ro, so, eid, sf, ridx, **kw)
            fn = lambda: bsq.grouped_quantize(x, args.fmt, ro, so, eid, sf, ridx, out=out, scales=sc, **kw)
    elif args.case == "gemm_quantize":
        # NVFP4 quantize fused into the epilogue of 8192 x 2048 x 7168
        x = to_dev_bf16(wl.config_dense_nvfp4_large()["x_bits"], device)
        wgt = x[4096:6144]
        out, sc = bsq.gemm_quantize(x, wgt, "nvfp4", 1.0)
        fn = lambda: bsq.gemm_quantize(x, wgt, "nvfp4", 1.0, out=out, scales=sc)
    elif args.case == "tensor_sf":
        x = to_dev_bf16(wl.config_dense_nvfp4_large()["x_bits"], device)
        ws = torch.zeros(bsq.lib().bsq_tensor_sf_workspace_bytes(), dtype=torch.uint8, device=device)
        out = bsq.tensor_sf(x, workspace=ws)
        fn = lambda: bsq.tensor_sf(x, out=out, workspace=ws)
    else:
        x = to_dev_bf16(wl.config_dense_mx_wide()["x_bits"], device)
        out, sc = bsq.quantize(x, args.case)
        fn = lambda: bsq.quantize(x, args.case, out=out, scales=sc)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_hold(1.0 + 0.2 * args.steps)
    a.record()
    for _ in range(args.steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    err = bsq.device_error()
    print(json.dumps({"case": args.case, "steps": args.steps, "warmup": args.warmup,
                      "us_per_launch": round(a.elapsed_time(b) * 1e3 / args.steps, 2),
                      "device_error": err}))
    if err:
        sys.exit(1)


def relaunch_ranks(n: int, argv) -> int:
    """Start this script as n ranks on this node (one per GPU) through
    torch.distributed.run on 127.0.0.1 and return its exit status."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the context workloads")
    ap.add_argument("--grouped-kernel", choices=("auto", "stream", "latency", "token"), default="auto",
                    help="kernel of the grouped --case workloads")
    ap.add_argument("--grouped-workspace", action="store_true",
                    help="with --case grouped_*: pass the scale-staging workspace")
    ap.add_argument("--fmt", choices=("nvfp4", "mxfp4", "mxfp8"), default="nvfp4",
                    help="format of the grouped --case workloads")
    ap.add_argument("--case", choices=CASES, default=None,
                    help="time one context workload alone on GPU 0 (for profiling) and exit")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.case is not None:
        run_case(args)
        return
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(relaunch_ranks(args.gpus, sys.argv[1:] if argv is None else list(argv)))
    rank, world, local_rank = dist_env()
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} does not match the {world} rank(s) of this launch (WORLD_SIZE)")
    print(f"bench: rank {rank} of {world} (local rank {local_rank}), impl {args.impl}", file=sys.stderr,
          flush=True)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
