"""Benchmark of the fused sublayer boundary on GB300.

One step = one decoder layer's two boundaries on a batch of T = 16384 tokens
(8 x 2048 prefill), D = 5120: the attention boundary (dense, n = 7) and the
MoE boundary (top-8 combine, n = 20). Together they run every step of the hot
path (combine, post-norm, depth-scaled residual, pre-norm).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). `value` is tokens/s through the step, all ranks
together (each rank has its own 16384-token batch: weak scaling, no
data-path collective). `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

T_TOKENS = 16384
D = 5120
DENSE_N, MOE_N, EPS = 7, 20, 1e-6
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
METRIC = "fused boundary tokens/s at T=16384 (dense + MoE boundary of one decoder layer)"
WORKLOAD = (f"layer boundary pair, T={T_TOKENS} tokens per GPU, D={D}: dense boundary n={DENSE_N} + "
            f"MoE top-8 combine boundary n={MOE_N}, eps=1e-6; storage bf16, math fp32")

# DRAM traffic per launch from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), valid only for the kernel source it was taken on.
NCU_TRAFFIC = {
    "moe": {"bytes_per_launch": 1_511_092_480 + 300_573_440, "source_sha": "b6b335c48b9cdff0"},
    "dense": {"bytes_per_launch": 335_653_376 + 264_058_624, "source_sha": "b6b335c48b9cdff0"},
}

# Routing is bound by instruction issue, not HBM: its warp-instructions per
# launch at T = 16384 (ncu smsp__inst_executed.sum) give its issue roofline,
# valid while the kernel source matches.
ROUTE_ISSUE = {"warp_instructions_per_launch": 11_224_712, "source_sha": "b6b335c48b9cdff0"}


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sandwich_norm_residual_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dense_bytes(T: int) -> int:
    return T * 8 * D + 4 * D           # read h, x; write h', y; two weight vectors


def moe_bytes(T: int) -> int:
    return T * (22 * D + 32) + 4 * D   # read 8 expert rows, 8 weights, h; write h', y


# ------------------------------------------------------------------ distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, device=None) -> float:
    """Max of a float over all ranks (one tiny all-reduce; identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def shard_rows(total: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous row block of `rank` (used when a fixed batch is split across ranks)."""
    per, rem = divmod(total, world)
    lo = rank * per + min(rank, rem)
    return lo, lo + per + (1 if rank < rem else 0)


# ------------------------------------------------------------------ clocks

class NvmlClockSampler:
    """SM clock, its maximum and the clock event (throttle) reasons, polled through
    NVML (libnvidia-ml, query calls only: nothing is set) every ~1 ms from a thread,
    so that a timed region of a few milliseconds still holds samples."""
    NAMES = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
             0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_id: str | None, index: int):
        import ctypes
        self.rows: list[tuple[float, float, float, int]] = []
        self.ok = False
        self._stop = threading.Event()
        self.t = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            rc = (lib.nvmlDeviceGetHandleByUUID(gpu_id.encode(), ctypes.byref(h)) if gpu_id
                  else lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)))
            if rc != 0:
                return
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.lib, self.h, self.ct = lib, h, ctypes
            mx = ctypes.c_uint(0)  # the maximum SM clock does not change: read it once
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:  # NVML_CLOCK_SM
                return
            self.max_mhz = float(mx.value)
            self.ok = self._poll() is not None
        except (OSError, AttributeError):
            self.ok = False

    def _poll(self):
        ct = self.ct
        mhz, rs = ct.c_uint(0), ct.c_ulonglong(0)
        if (self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) != 0 or  # NVML_CLOCK_SM
                self.reasons_fn(self.h, ct.byref(rs)) != 0):
            return None
        return float(mhz.value), self.max_mhz, int(rs.value)

    def _run(self):
        while not self._stop.is_set():
            r = self._poll()
            if r is not None:
                self.rows.append((time.time(),) + r)
            time.sleep(0.001)

    def start(self):
        self.t = threading.Thread(target=self._run, daemon=True)
        self.t.start()

    def stop(self):
        self._stop.set()
        if self.t:
            self.t.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [r for r in self.rows if t0 <= r[0] <= t1]
        mhz = sorted(r[1] for r in inside)
        reasons = set()
        for r in inside:
            reasons |= {n for bit, n in self.NAMES.items() if r[3] & bit}
        return {"sm_mhz": mhz[len(mhz) // 2] if mhz else None,
                "sm_max_mhz": inside[-1][2] if inside else None, "reasons": sorted(reasons),
                "samples": len(inside), "source": "nvml, ~1 ms polling"}


class ClockSampler:
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.rows: list[tuple[float, list[str]]] = []
        self.proc = None
        self.gpu_id = gpu_id
        self.t = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [r for (t, r) in self.rows if t0 <= t <= t1]
        used = inside or [r for (t, r) in self.rows if t >= t0][:3]
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in used:
            try:
                mhz.append(float(r[1]))
                mx = float(r[2])
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        mhz.sort()
        return {"sm_mhz": mhz[len(mhz) // 2] if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(inside)}


# ------------------------------------------------------------------ our arm

def measured_hbm_peak() -> tuple[float, str]:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def make_inputs(device, pin: bool):
    import torch
    import synth
    from synth import DENSE_PREFILL_T16384, MOE_T16384
    dense_cfg, moe_cfg = DENSE_PREFILL_T16384, MOE_T16384
    dn = synth.dense_inputs(dense_cfg)
    mo = synth.moe_inputs(moe_cfg)
    host = {"dense": dn, "moe": mo}
    if pin:
        host = {g: {k: v.pin_memory() for k, v in d.items()} for g, d in host.items()}
    dev = {g: {k: v.to(device) for k, v in d.items()} for g, d in host.items()}
    dev["dense"]["y"] = torch.empty_like(dev["dense"]["h"])
    dev["moe"]["y"] = torch.empty_like(dev["moe"]["h"])
    return host, dev


def run_step(snr, d, stream, pdl: bool = False):
    """One step: the dense then the MoE boundary. With pdl, each kernel is a
    programmatic dependent launch: it stages its norm weights while the previous
    kernel on the stream finishes (their weight buffers are disjoint)."""
    dn, mo = d["dense"], d["moe"]
    opts = dict(flags=snr._lib.BEAM_OPT_PDL) if pdl else None
    snr.boundary_fused(dn["h"], dn["x"], dn["post_w"], dn["pre_w"], DENSE_N, EPS, y=dn["y"],
                       stream=stream, opts=opts)
    snr.moe_combine_boundary(mo["h"], mo["expert_out"], mo["topk_w"], mo["post_w"], mo["pre_w"],
                             MOE_N, EPS, y=mo["y"], stream=stream, opts=opts)


def decode_latency(snr, device, replays: int = 20) -> dict:
    """Decode-size boundaries, launch-bound: CUDA-graph replays, with and without
    programmatic dependent launch (PDL). T = 4: microseconds per boundary over
    200 captured calls. T = 64: microseconds per 104-boundary chain (n = 2..105,
    fresh x and weights per boundary), of dense boundaries only and of dense and
    MoE boundaries in turn as a decoder's 52 layers run them; and per-head Q/K
    norm with RoPE at T = 64, microseconds per layer over 52 captured launches."""
    import torch
    import synth
    from synth import DECODE_CHAIN_T64, DENSE_DECODE_T4, MOE_T16384
    out = {}
    stream = torch.cuda.Stream(device)
    pdl_opts = {False: None, True: dict(flags=snr._lib.BEAM_OPT_PDL)}

    def timed_graph(body, label, reps):
        with torch.cuda.stream(stream):
            body()  # first calls set up the launch shapes outside the capture
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):  # replays run on the current stream
            g.replay()
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) * 1e3 / reps

    c0 = DENSE_DECODE_T4
    d0 = {k: v.to(device) for k, v in synth.dense_inputs(c0).items()}
    y0 = torch.empty_like(d0["h"])
    for pdl in (False, True):
        def body0(pdl=pdl):
            for _ in range(200):
                snr.boundary_fused(d0["h"], d0["x"], d0["post_w"], d0["pre_w"], c0.n, c0.eps, y=y0,
                                   opts=pdl_opts[pdl], stream=stream)
        out[f"T4_us_per_boundary{'_pdl' if pdl else ''}"] = timed_graph(body0, "t4", replays) / 200

    c1 = DECODE_CHAIN_T64
    h1 = synth.dense_inputs(c1)["h"].to(device)
    steps = [{k: v.to(device) for k, v in synth.dense_inputs(c1, step=s).items()}
             for s in range(c1.steps)]
    ys = torch.empty((c1.steps,) + tuple(h1.shape), dtype=h1.dtype, device=device)
    for pdl in (False, True):
        def body1(pdl=pdl):
            for s, d in enumerate(steps):
                snr.boundary_fused(h1, d["x"], d["post_w"], d["pre_w"], c1.n + s, c1.eps, y=ys[s],
                                   opts=pdl_opts[pdl], stream=stream)
        out[f"chain104_T64_us{'_pdl' if pdl else ''}"] = timed_graph(body1, "chain", replays)
    # the chain as a decoder runs it: attention (dense) and MoE boundaries in turn
    from synth import layer_chain_inputs
    _, lsteps = layer_chain_inputs(c1, MOE_T16384)
    lsteps = [{k: (v.to(device) if k != "kind" else v) for k, v in st.items()} for st in lsteps]
    for pdl in (False, True):
        def body2(pdl=pdl):
            for s, d in enumerate(lsteps):
                if d["kind"] == "dense":
                    snr.boundary_fused(h1, d["x"], d["post_w"], d["pre_w"], c1.n + s, c1.eps,
                                       y=ys[s], opts=pdl_opts[pdl], stream=stream)
                else:
                    snr.moe_combine_boundary(h1, d["expert_out"], d["topk_w"], d["post_w"],
                                             d["pre_w"], c1.n + s, c1.eps, y=ys[s],
                                             opts=pdl_opts[pdl], stream=stream)
        out[f"layer_chain104_T64_us{'_pdl' if pdl else ''}"] = timed_graph(body2, "layers", replays)
    # per-head Q/K norm with RoPE at T = 64, one launch per layer (52), in place
    import numpy as np
    q64 = torch.from_numpy((synth.normal(1, 10, 64 * QK_HEADS * QK_DIM) * 2.0)
                           .reshape(64, QK_HEADS, QK_DIM)).to(device).to(torch.bfloat16)
    k64 = torch.from_numpy((synth.normal(1, 11, 64 * QK_KV_HEADS * QK_DIM) * 2.0)
                           .reshape(64, QK_KV_HEADS, QK_DIM)).to(device).to(torch.bfloat16)
    qw64 = torch.from_numpy(1 + 0.1 * synth.normal(1, 12, QK_DIM)).to(device).to(torch.bfloat16)
    kw64 = torch.from_numpy(1 + 0.1 * synth.normal(1, 13, QK_DIM)).to(device).to(torch.bfloat16)
    pos64 = torch.arange(1000, 1064, dtype=torch.int32, device=device)
    inv = 10000.0 ** (-np.arange(0, QK_DIM, 2) / QK_DIM)
    ang = np.arange(QK_SEQ)[:, None] * inv[None, :]
    tab = torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], 1).astype(np.float32)).to(device)
    for pdl in (False, True):
        def body3(pdl=pdl):
            for _ in range(52):
                snr.qk_norm(q64, k64, qw64, kw64, pos64, 1e-6, "rope", rope_table=tab, stream=stream,
                            pdl=pdl)
        out[f"qk_norm_rope_T64_us_per_layer{'_pdl' if pdl else ''}"] = timed_graph(body3, "qk", replays) / 52
    # top-8 routing at T = 64, one launch per layer (52)
    z64 = torch.from_numpy((synth.normal(1, 8, 64 * 256) * 2.0).reshape(64, 256)).to(device)
    b64 = torch.from_numpy(synth.normal(1, 9, 256) * 0.05).to(device)
    i64 = torch.empty((64, 8), dtype=torch.int32, device=device)
    w64 = torch.empty((64, 8), dtype=torch.float32, device=device)

    for pdl in (False, True):
        def body4(pdl=pdl):
            for _ in range(52):
                snr.moe_route(z64, b64, idx=i64, w=w64, stream=stream, pdl=pdl)
        out[f"route_T64_us_per_layer{'_pdl' if pdl else ''}"] = timed_graph(body4, "route", replays) / 52
    # the dense chain launched one call at a time, no graph
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(replays):
            for s, d in enumerate(steps):
                snr.boundary_fused(h1, d["x"], d["post_w"], d["pre_w"], c1.n + s, c1.eps, y=ys[s],
                                   stream=stream)
        b.record(stream)
    torch.cuda.synchronize(device)
    out["chain104_T64_us_stream_launches"] = a.elapsed_time(b) * 1e3 / replays
    snr.sync_status(stream)
    return {k: round(v, 2) for k, v in out.items()}


def nvfp4_bytes(T: int, moe: bool) -> int:
    # as the BF16 boundaries, with y written as D/2 code bytes + D/16 scale bytes
    y_bf16, y_fp4 = 2 * D, D // 2 + D // 16
    return (moe_bytes(T) if moe else dense_bytes(T)) - T * y_bf16 + T * y_fp4


QK_HEADS, QK_KV_HEADS, QK_DIM, QK_SEQ = 48, 8, 128, 2048


def qk_bytes(T: int, rope: bool) -> int:
    # q and k read and written in place, one position per token, the two weight
    # vectors; RoPE also reads the cos|sin table once (2048 positions x 128 FP32)
    b = T * ((QK_HEADS + QK_KV_HEADS) * QK_DIM * 2 * 2 + 4) + 2 * QK_DIM * 2
    return b + (QK_SEQ * QK_DIM * 4 if rope else 0)


def route_bytes(T: int) -> int:
    return T * (256 * 4 + 8 * 8) + 256 * 4   # FP32 logits in; ids and weights out; bias


MIN_LAUNCHES, MIN_SECONDS = 1000, 0.5


def _time_loop(fn, stream, reps: int) -> float:
    import torch
    with torch.cuda.stream(stream):
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(reps):
            fn(i)
        e.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(e) * 1e3 / reps


def _time_launches(fn, stream, reps: int | None = None, warmup: int = 3) -> tuple[float, int]:
    """Mean microseconds per launch over back-to-back launches, CUDA events on the
    launching stream: `reps` launches, or by default at least MIN_LAUNCHES and at
    least MIN_SECONDS of launches (sized from a 20-launch estimate). Returns
    (us, launches)."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fn(i)
    torch.cuda.synchronize()
    if reps is None:
        est = _time_loop(fn, stream, 20)
        reps = max(MIN_LAUNCHES, int(MIN_SECONDS / (est * 1e-6)) + 1)
    return _time_loop(fn, stream, reps), reps


def next_rows(snr, device, dev, peak: float, sm_mhz: float | None = None) -> dict:
    """The scope table's next rows at T = 16384, each timed on its own and
    reported beside the step (none is part of it): group-limited top-8 routing,
    per-head Q/K norm with RoPE or SSMax (8 sequences of 2048 positions), and
    the two boundaries with y written as NVFP4. Routing also reports its issue
    roofline: 4 warp-instructions per SM per clock at `sm_mhz`."""
    import torch
    import synth
    stream = torch.cuda.Stream(device)
    T = T_TOKENS
    out = {}

    def entry(us, nbytes):
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"us": round(us, 2), "bytes": nbytes, "GBps": round(gbs, 1),
                "frac_of_measured_hbm": round(gbs / peak, 4)}

    # routing: ten logit buffers in turn, so each launch reads from DRAM (L2 holds one)
    nbuf = 10
    z = torch.from_numpy((synth.normal(3, 8, nbuf * T * 256) * 2.0).reshape(nbuf, T, 256)).to(device)
    b = torch.from_numpy(synth.normal(3, 9, 256) * 0.05).to(device)
    idx = torch.empty((T, 8), dtype=torch.int32, device=device)
    w = torch.empty((T, 8), dtype=torch.float32, device=device)
    us, n_rt = _time_launches(lambda i: snr.moe_route(z[i % nbuf], b, idx=idx, w=w, stream=stream),
                              stream)
    rt = entry(us, route_bytes(T))
    rt["launches"] = n_rt
    if sm_mhz and ROUTE_ISSUE["source_sha"] == kernel_source_sha():
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        issue_peak = sms * 4 * sm_mhz * 1e6  # warp-instructions per second
        inst = ROUTE_ISSUE["warp_instructions_per_launch"]
        rt.update({"bound": "issue", "warp_instructions": inst, "issue_peak_per_s": issue_peak,
                   "frac_of_issue_peak": round(inst / (us * 1e-6) / issue_peak, 4)})
    out["route_top8_of_256"] = rt
    del z

    # Q/K norm: q [T, 48, 128] and k [T, 8, 128] (235 MB together, above L2)
    q = torch.from_numpy((synth.normal(3, 10, T * QK_HEADS * QK_DIM) * 2.0)
                         .reshape(T, QK_HEADS, QK_DIM)).to(device).to(torch.bfloat16)
    k = torch.from_numpy((synth.normal(3, 11, T * QK_KV_HEADS * QK_DIM) * 2.0)
                         .reshape(T, QK_KV_HEADS, QK_DIM)).to(device).to(torch.bfloat16)
    qw = torch.from_numpy(1 + 0.1 * synth.normal(3, 12, QK_DIM)).to(device).to(torch.bfloat16)
    kw = torch.from_numpy(1 + 0.1 * synth.normal(3, 13, QK_DIM)).to(device).to(torch.bfloat16)
    pos = (torch.arange(T, dtype=torch.int32, device=device) % QK_SEQ).contiguous()
    inv = 10000.0 ** (-torch.arange(0, QK_DIM, 2, dtype=torch.float64) / QK_DIM)
    ang = torch.arange(QK_SEQ, dtype=torch.float64)[:, None] * inv[None, :]
    table = torch.cat([ang.cos(), ang.sin()], 1).float().to(device).contiguous()
    for mode in ("rope", "ssmax"):
        us, nl = _time_launches(lambda i, mode=mode: snr.qk_norm(
            q, k, qw, kw, pos, 1e-6, mode=mode, rope_table=table if mode == "rope" else None,
            stream=stream), stream)
        out[f"qk_norm_{mode}"] = dict(entry(us, qk_bytes(T, mode == "rope")), launches=nl)
    del q, k

    # the boundaries with y as NVFP4, on the step's own buffers
    dn, mo = dev["dense"], dev["moe"]
    gs = 336.0
    yq = torch.empty((T, D // 2), dtype=torch.uint8, device=device)
    ys = torch.empty((T, D // 16), dtype=torch.uint8, device=device)
    us, nl = _time_launches(lambda i: snr.boundary_fused_nvfp4(
        dn["h"], dn["x"], dn["post_w"], dn["pre_w"], DENSE_N, EPS, gs, y_fp4=yq, y_scale=ys,
        stream=stream), stream)
    out["dense_boundary_nvfp4"] = dict(entry(us, nvfp4_bytes(T, False)), launches=nl)
    us, nl = _time_launches(lambda i: snr.moe_combine_boundary_nvfp4(
        mo["h"], mo["expert_out"], mo["topk_w"], mo["post_w"], mo["pre_w"], MOE_N, EPS, gs,
        y_fp4=yq, y_scale=ys, stream=stream), stream)
    out["moe_boundary_nvfp4"] = dict(entry(us, nvfp4_bytes(T, True)), launches=nl)
    snr.sync_status(stream)
    return out


def moe_stress(snr, device, peak: float, reps: int = 5) -> dict:
    """The MoE stress workload at full size: T = 131072 tokens, n = 104, Student-t(3)
    expert rows with 0.1% of them x100, one launch of 14.8 GB of algorithmic traffic.
    Inputs are generated in chunks straight into device memory."""
    import torch
    import synth
    from synth import MOE_STRESS_T131072
    cfg = MOE_STRESS_T131072
    T, D, K = cfg.T, cfg.D, cfg.K
    e = torch.empty((T, K, D), dtype=torch.bfloat16, device=device)
    for r in range(0, T, 8192):
        e[r:r + 8192].copy_(synth.expert_rows(cfg, r, min(8192, T - r)))
    h = synth.to_bf16(synth.normal(cfg.seed, synth.STREAMS["h"], T * D).reshape(T, D)).to(device)
    w = torch.from_numpy(synth.topk_weights(cfg.seed, synth.STREAMS["topk"], T, K,
                                            cfg.route_scale)).to(device)
    pw = synth.to_bf16(synth.normal(cfg.seed, synth.STREAMS["post_w"], D, 0, 0.1, 1.0)).to(device)
    qw = synth.to_bf16(synth.normal(cfg.seed, synth.STREAMS["pre_w"], D, 0, 0.1, 1.0)).to(device)
    y = torch.empty_like(h)
    stream = torch.cuda.Stream(device)
    us, _ = _time_launches(lambda i: snr.moe_combine_boundary(h, e, w, pw, qw, cfg.n, cfg.eps, y=y,
                                                              stream=stream), stream, reps, warmup=2)
    snr.sync_status(stream)
    nbytes = T * (22 * D + 32) + 4 * D
    gbs = nbytes / (us * 1e-6) / 1e9
    del e, h, w, y
    torch.cuda.empty_cache()
    return {"T": T, "n": cfg.n, "us": round(us, 1), "bytes": nbytes, "GBps": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peak, 4), "tokens_per_s": T / (us * 1e-6)}


def bench_ours(args, rank, world, local_rank):
    import torch
    import sandwich_norm_residual_gb300 as snr
    from sandwich_norm_residual_gb300 import build as libbuild

    libbuild.build()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    stream = torch.cuda.Stream(device)
    host, dev = make_inputs(device, pin=True)

    pdl = not args.no_pdl
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            run_step(snr, dev, stream, pdl)
    snr.sync_status(stream)

    try:
        props = torch.cuda.get_device_properties(device)
        uuid = str(getattr(props, "uuid", "") or "")
        gpu_id = f"GPU-{uuid}" if uuid and not uuid.startswith("GPU-") else (uuid or None)
    except Exception:
        gpu_id = None
    sampler = NvmlClockSampler(gpu_id, local_rank)
    if not sampler.ok:
        sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize(device)
    t0 = time.time()
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(args.steps):
            run_step(snr, dev, stream, pdl)
        end.record(stream)
    torch.cuda.synchronize(device)
    t1 = time.time()
    barrier(device)
    snr.sync_status(stream)

    # per-kernel durations, for the roofline: each kernel alone, back to back on
    # the launching stream (plain launches), CUDA events around the whole loop;
    # at least MIN_LAUNCHES launches and MIN_SECONDS whatever --steps is
    dn, mo = dev["dense"], dev["moe"]
    k0 = time.time()
    dense_us, dense_n = _time_launches(lambda i: snr.boundary_fused(
        dn["h"], dn["x"], dn["post_w"], dn["pre_w"], DENSE_N, EPS, y=dn["y"], stream=stream), stream)
    moe_us, moe_n = _time_launches(lambda i: snr.moe_combine_boundary(
        mo["h"], mo["expert_out"], mo["topk_w"], mo["post_w"], mo["pre_w"], MOE_N, EPS, y=mo["y"],
        stream=stream), stream)
    k1 = time.time()
    snr.sync_status(stream)
    time.sleep(0.05)
    sampler.stop()

    ms_total = start.elapsed_time(end)
    ms_total = max_over_ranks(ms_total, device)
    ms_step = ms_total / args.steps

    # end to end through the public API with the batch in host memory: page-locked
    # inputs and outputs that the kernels read and write over the CPU-GPU link
    # (beam_*_host); h' overwrites h in host memory, y lands in host memory
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    y_host = {g: torch.empty(host[g]["h"].shape, dtype=torch.bfloat16, pin_memory=True)
              for g in ("dense", "moe")}
    h2d = sum(v.numel() * v.element_size() for g in host.values() for v in g.values())
    d2h = sum(2 * y.numel() * y.element_size() for y in y_host.values())   # h' and y

    def host_step():
        hd, hm = host["dense"], host["moe"]
        snr.boundary_fused_host(hd["h"], hd["x"], hd["post_w"], hd["pre_w"], DENSE_N, EPS,
                                y=y_host["dense"], stream=stream)
        snr.moe_combine_boundary_host(hm["h"], hm["expert_out"], hm["topk_w"], hm["post_w"],
                                      hm["pre_w"], MOE_N, EPS, y=y_host["moe"], stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(2):
            host_step()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            host_step()
        e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, device)
    snr.sync_status(stream)

    # for comparison: copy the inputs in, run the device calls, copy h' and y out
    out_host = {g: {k: torch.empty_like(host[g]["h"], device="cpu").pin_memory() for k in ("h", "y")}
                for g in ("dense", "moe")}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            for g in ("dense", "moe"):
                for k, v in host[g].items():
                    dev[g][k].copy_(v, non_blocking=True)
            run_step(snr, dev, stream)
            for g in ("dense", "moe"):
                for k in ("h", "y"):
                    out_host[g][k].copy_(dev[g][k], non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize(device)
    copy_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, device)
    snr.sync_status(stream)

    if rank != 0:
        _finish(world)
        return

    peak, peak_kind = measured_hbm_peak()
    db, mb = dense_bytes(T_TOKENS), moe_bytes(T_TOKENS)
    dense_gbs = db / (dense_us * 1e-6) / 1e9
    moe_gbs = mb / (moe_us * 1e-6) / 1e9
    sha = kernel_source_sha()
    tr = NCU_TRAFFIC.get("moe")
    traffic = tr["bytes_per_launch"] if tr and tr.get("source_sha") == sha else None
    clocks = sampler.summary(t0, t1)
    clocks["per_kernel_loops"] = sampler.summary(k0, k1)
    line = {
        "metric": METRIC,
        "value": world * T_TOKENS / (ms_step * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": WORKLOAD,
            "T": T_TOKENS, "D": D,
            "l2": "inputs larger than L2 (129 MB): no flush between steps",
            "step": ("dense then MoE boundary per step, programmatic dependent launches (each "
                     "kernel stages its weights while the previous one finishes)" if pdl else
                     "dense then MoE boundary per step, plain launches"),
            "per_kernel": (f"each kernel alone, back-to-back plain launches (at least {MIN_LAUNCHES} "
                           f"and {MIN_SECONDS} s: dense {dense_n}, MoE {moe_n}), CUDA events"),
            "dense": {"us": dense_us, "tokens_per_s": T_TOKENS / (dense_us * 1e-6),
                      "GBps": dense_gbs, "frac_of_measured_hbm": dense_gbs / peak,
                      "frac_of_nominal_8TBps": dense_gbs / NOMINAL_HBM_GBS, "bytes": db},
            "moe": {"us": moe_us, "tokens_per_s": T_TOKENS / (moe_us * 1e-6),
                    "GBps": moe_gbs, "frac_of_measured_hbm": moe_gbs / peak,
                    "frac_of_nominal_8TBps": moe_gbs / NOMINAL_HBM_GBS, "bytes": mb},
            "kernel_source_sha": sha,
            "parallelism": f"{world} independent replica(s), no collective on the data path",
        },
        "roofline": {"kernel": "moe_combine_boundary", "bound": "hbm", "achieved": moe_gbs,
                     "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                     "frac": moe_gbs / peak, "traffic": traffic},
        "e2e": {"value": world * T_TOKENS / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "ms_per_step": e2e_ms,
                "path": "beam_boundary_fused_host + beam_moe_combine_boundary_host on page-locked "
                        "host buffers: the kernels read the inputs and write h' and y over the "
                        "CPU-GPU link",
                "copy_then_compute": {"value": world * T_TOKENS / (copy_ms * 1e-3),
                                      "ms_per_step": copy_ms}},
        "gpu_launches": 2 * args.steps,  # in the timed region
        "clocks": clocks,
    }
    if not args.no_decode:
        line["config"]["decode"] = decode_latency(snr, device)
    if not args.no_next_rows:
        line["config"]["next_rows"] = next_rows(snr, device, dev, peak,
                                                clocks.get("sm_mhz") or clocks.get("sm_max_mhz"))
    if not args.no_stress:
        line["config"]["moe_stress_T131072"] = moe_stress(snr, device, peak)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    print(json.dumps(line), flush=True)
    _finish(world)


def _finish(world):
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ oracle timing

def oracle_step_sample(rows: int, row0: int = 0):
    """Inputs of `rows` tokens of the step's workload (both boundaries)."""
    import synth
    from synth import DENSE_PREFILL_T16384, MOE_T16384
    return (synth.dense_inputs(DENSE_PREFILL_T16384, row_start=row0, rows=rows),
            synth.moe_inputs(MOE_T16384, row_start=row0, rows=rows))


def oracle_step(dn, mo, threads: int = 1):
    import oracle
    oracle.boundary(dn["h"], dn["x"], dn["post_w"], dn["pre_w"], DENSE_N, EPS, threads=threads)
    oracle.moe_boundary(mo["h"], mo["expert_out"], mo["topk_w"], mo["post_w"], mo["pre_w"], MOE_N,
                        EPS, threads=threads)


def _oracle_rate(seconds: float, threads: int) -> tuple[float, int, float]:
    rows, done, spent = 16 * threads, 0, 0.0
    while spent < seconds:
        dn, mo = oracle_step_sample(rows, done % T_TOKENS)
        t0 = time.perf_counter()
        oracle_step(dn, mo, threads)
        spent += time.perf_counter() - t0
        done += rows
    return done / spent, done, spent


def cpu_baseline(seconds: float) -> dict:
    """The oracle, as it stands, on one host core, over a bounded sample of the workload;
    beside it the same oracle row-parallel on every host core."""
    rate, done, spent = _oracle_rate(seconds, 1)
    line = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of the {T_TOKENS} tokens through both boundaries, "
                      f"{spent:.1f} s single-threaded C"}
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    if cores > 1:
        rate_n, done_n, spent_n = _oracle_rate(seconds / 2, cores)
        line["all_cores"] = {"value": rate_n, "unit": "tokens/s", "cores": cores,
                             "sample": f"{done_n} tokens, {spent_n:.1f} s, rows split over {cores} "
                                       "threads"}
    return line


def bench_reference(args, rank, world):
    if rank != 0:
        return
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_step(*oracle_step_sample(rows))
    spent = 0.0
    for i in range(args.steps):
        dn, mo = oracle_step_sample(rows, (i * rows) % T_TOKENS)
        t0 = time.perf_counter()
        oracle_step(dn, mo)
        spent += time.perf_counter() - t0
    value = args.steps * rows / spent
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * spent / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T_TOKENS, "D": D,
                   "sample": f"each step runs {rows} of the workload's tokens through both boundaries"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows} tokens per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-rows", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode-size latency figures")
    ap.add_argument("--no-pdl", action="store_true",
                    help="plain launches in the timed step instead of programmatic dependent ones")
    ap.add_argument("--no-stress", action="store_true",
                    help="skip the T = 131072 MoE stress timing")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the timings of routing, Q/K norm and the NVFP4 boundaries")
    args = ap.parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        bench_reference(args, rank, world)
    else:
        bench_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
