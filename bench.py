"""Benchmark of the selective-SSM serving step on GB300.

One step = the whole hot path over one batch of the long-context mixed
workload (8 fresh prefills of 65536 tokens plus 384 single-token decodes,
chunk 256, H=128, P=64, N=128, G=8, bf16 tokens, fp32 state cache of 16384
slots): host chunk metadata, its copy to the device, ssd_prefill_varlen,
ssm_decode_update.  Inputs are seeded synthetic tensors of that shape; the
inputs (8.6 GB of x alone) are larger than the 129 MB L2, so no flush is
needed between steps.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead, on
a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "SSD prefill tokens/s/layer and decode state-updates/s; % HBM roofline on 1 GB300"
UNIT = "tokens/s/layer"
WORKLOADS = {
    # the benchmark: every step of the path, long-context mixed batch
    "long_mixed": dict(workload="long-context mixed batch: 8 x 65536-token prefills + 384 single-token decodes",
                       num_prefills=8, prefill_len=65536, num_decodes=384, chunk_size=256, nheads=128,
                       headdim=64, dstate=128, ngroups=8, cache_slots=16384, token_dtype="bf16",
                       state_dtype="fp32", l2="inputs larger than L2 (no flush)"),
    # a smaller case of the same kernels for profiler captures (about 4 GB on the device)
    "prefill_8x8192": dict(workload="8 x 8192-token prefills (profiling size)", num_prefills=8, prefill_len=8192,
                           num_decodes=0, chunk_size=256, nheads=128, headdim=64, dstate=128, ngroups=8,
                           cache_slots=512, token_dtype="bf16", state_dtype="fp32",
                           l2="inputs larger than L2 (no flush)"),
    # the decode kernel at the long batch's request count, on a smaller cache (about 4 GB) for captures
    "decode_384": dict(workload="384 single-token decodes on a 1024-slot cache, one 256-token prefill (profiling size)",
                       num_prefills=1, prefill_len=256, num_decodes=384, chunk_size=256, nheads=128, headdim=64,
                       dstate=128, ngroups=8, cache_slots=1024, token_dtype="bf16", state_dtype="fp32",
                       l2="state reads larger than L2 (no flush)"),
}
WORKLOAD = WORKLOADS["long_mixed"]


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _bf16_peak():
    """Dense bf16 tensor TFLOP/s for a kernel timed on its own (the burst figure); fp16 operands
    run at the same rate."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst)"
    except Exception:
        return 1900.0, "fallback"


def _sm_max_mhz():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["sm_max_mhz"])
    except Exception:
        return SM_MAX_MHZ


# ------------------------------------------------------------- byte counts --

# DRAM traffic of one prefill call (tensor-core path, no segment split), from one ncu capture of both
# its kernels on 8 x 8192 tokens at H=128, P=64, N=128, G=8, chunk 256: prep_kernel 285,258,752 B read +
# 286,390,528 B written; ssd_prefill_tc_kernel 1,424,511,488 B read + 2,090,916,864 B written.  Scaled by
# tokens (x, y, B/C, delta and one state per 256-token chunk all grow with them).  Only for that head
# configuration and this kernel version; the summary is in profiles/.
FUSED_TRAFFIC_PER_TOKEN = (1424511488 + 2090916864) / 65536
PREFILL_TRAFFIC_PER_TOKEN = (285258752 + 286390528) / 65536 + FUSED_TRAFFIC_PER_TOKEN
PREFILL_TRAFFIC_SOURCE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of prep_kernel and ssd_prefill_tc_kernel "
                          "on 8 x 8192 tokens, scaled by tokens")
FUSED_TRAFFIC_SOURCE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of ssd_prefill_tc_kernel on 8 x 8192 "
                        "tokens, scaled by tokens")
SM_MAX_MHZ = 2070.0  # GB300's maximum SM clock, where the measured-peaks file does not give it


def prefill_traffic(T, H, P, N, G, fused_only=False):
    if (H, P, N, G) != (128, 64, 128, 8):
        return None
    return (FUSED_TRAFFIC_PER_TOKEN if fused_only else PREFILL_TRAFFIC_PER_TOKEN) * T


def prefill_bytes(T, K, H, P, N, G, elt, init_reads=0):
    """Algorithmic HBM bytes of one prefill call: x in, y out, dt, B, C per
    token; one fp32 state store per chunk; one state load per initial state."""
    per_tok = 2 * H * P * elt + H * elt + 2 * G * N * elt
    return T * per_tok + (K + init_reads) * H * P * N * 4


def fused_bytes(T, K, H, P, N, G, elt, init_reads=0):
    """The fused kernel's share of the call's algorithmic bytes: all of them but dt, which the prep
    kernel reads (the fused kernel reads its delta and cumsum instead)."""
    return prefill_bytes(T, K, H, P, N, G, elt, init_reads) - T * H * elt


# The fused prefill cuts every chunk into blocks of at most 128 tokens and issues, per block and
# head, four dense products on full 128-row tiles: S = C B^T (128 x 128, K = N), Y1 = P X
# (128 x P, K = 128), Y2 = C Hprev^T (128 x P, K = N) and dS = B^T (w x) (N x P, K = 128).
TC_BLOCK = 128


def prefill_method_flops(T, H, P, N, G, Q=TC_BLOCK):
    """The method's own flops at internal block Q: per token G Q N (the causal half of C B^T per
    group), H Q P (its causal product with delta x per head) and 4 H P N (the chunk-state update and
    C . h_prev) -- no masked halves, no per-head recomputation of C B^T."""
    return T * (G * Q * N + H * Q * P + 4 * H * P * N)


def prefill_mma_flops(cu_chunk_seqlens, H, P, N):
    """Tensor-core flops one fused prefill call issues (the masked upper half of S and P included)."""
    lens = np.diff(np.asarray(cu_chunk_seqlens, dtype=np.int64))
    blocks = int(((lens + TC_BLOCK - 1) // TC_BLOCK).sum())
    L = TC_BLOCK
    per_block_head = 2 * (L * L * N + L * P * L + L * P * N + N * P * L)
    return blocks * H * per_block_head


def decode_bytes(live, tpr, writes, H, P, N, G, elt):
    """One state load per live request, one state store per written column,
    plus the token tensors of the live rows."""
    per_tok = 2 * H * P * elt + H * elt + 2 * G * N * elt
    return (live + writes) * H * P * N * 4 + live * tpr * per_tok


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [v.strip() for v in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx.append(float(f[2]))
                except ValueError:
                    continue
                for name, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# -------------------------------------------------------------- GPU arm -----

class Step:
    """Holds one rank's device-resident workload and runs the step."""

    def __init__(self, dev, wl):
        import selective_state_space_mamba2_gb300 as ssd
        from selective_state_space_mamba2_gb300 import workloads as W
        self.ssd = ssd
        self.dev = dev
        self.pre, self.dec = W.long_mixed(dev, num_prefills=wl["num_prefills"], prefill_len=wl["prefill_len"],
                                          num_decodes=wl["num_decodes"], num_slots=wl["cache_slots"])
        p = self.pre
        self.H, self.P = p["x"].shape[1], p["x"].shape[2]
        self.G, self.N = p["B"].shape[1], p["B"].shape[2]
        self.y = torch.empty_like(p["x"])
        self.yd = torch.empty_like(self.dec["x"])
        self.cu_dev = p["cu_seqlens"].to(dev)
        self.si_dev = self.dec["state_indices"].to(dev)
        self.meta = self.metadata()
        self.K = len(self.meta["seq_idx"])
        m = self.device_meta(self.meta)
        a = ssd.prefill_args(p["x"], p["dt"], p["A"], p["B"], p["C"], self.cu_dev, m["cu_chunk_seqlens"],
                             m["seq_idx"], m["last_chunk_indices"], self.y, m["init_slot"], m["chunk_slot"],
                             p["cache"], p["D"], p["dt_bias"], chunk_size=p["chunk_size"], seq_order=m["seq_order"])
        self.workspace = torch.empty(max(ssd.ssd_prefill_workspace_size(a), 1), dtype=torch.uint8, device=dev)
        self.prefill_kernels = ssd.ssd_prefill_kernel_count(a)
        # The timed steps are issued on a stream of their own (not the legacy default stream,
        # which would serialise with every other stream); ssd_mixed_step forks the two parts of a
        # mixed step onto the library's own prioritised streams and joins them back into it.
        self.stream = torch.cuda.Stream(device=dev)

    def metadata(self):
        p = self.pre
        return self.ssd.ssd_chunk_metadata(p["cu_seqlens"], p["chunk_size"], p["num_computed"], p["has_init"],
                                           block_table=p["block_table"], null_block_id=p["null_block_id"])

    def device_meta(self, meta):
        """The metadata on the device, copied from pinned staging buffers (a copy from pageable
        memory would hold the host thread until the stream reaches it).  The staging buffers are
        reused every step; the bench's metadata is the same every step, so refilling one while an
        earlier step's copy from it is still queued cannot change what that copy reads."""
        if not hasattr(self, "_pin"):
            self._pin = {}
        out = {}
        for k, v in meta.items():
            t = torch.from_numpy(v)
            if k not in self._pin or self._pin[k].numel() < t.numel():
                self._pin[k] = torch.empty(max(t.numel(), 1), dtype=t.dtype, pin_memory=True)
            stage = self._pin[k][:t.numel()].view(t.shape)
            stage.copy_(t)
            out[k] = stage.to(self.dev, non_blocking=True)
        return out

    def run(self, ev=None, host=None, mixed=False, bufs=None):
        """One step on the current stream.  ev: optional (start, fused, mid, end) CUDA events: before
        the prefill call, at the library's mark before its fused kernel, between the calls and after
        the decode (serial step only).  host: pinned host buffers for the e2e
        leg.  mixed: both calls as one ssd_mixed_step (the decode beside the prefill).
        bufs: another set of device token buffers (x, dt, B, C of both calls and the outputs)."""
        p, d = dict(self.pre), dict(self.dec)
        y, yd = self.y, self.yd
        if bufs is not None:
            for name in ("x", "dt", "B", "C"):
                p[name], d[name] = bufs["p_" + name], bufs["d_" + name]
            y, yd = bufs["y"], bufs["yd"]
        if host is not None:  # end to end: this step's inputs come from host memory
            for name in ("x", "dt", "B", "C"):
                p[name].copy_(host["p_" + name], non_blocking=True)
                d[name].copy_(host["d_" + name], non_blocking=True)
        meta = self.metadata()
        m = self.device_meta(meta)
        if mixed and self.dec["live"] > 0:  # both parts in one library call (ssd_mixed_step)
            pa = self.ssd.prefill_args(p["x"], p["dt"], p["A"], p["B"], p["C"], self.cu_dev, m["cu_chunk_seqlens"],
                                       m["seq_idx"], m["last_chunk_indices"], y, m["init_slot"], m["chunk_slot"],
                                       p["cache"], p["D"], p["dt_bias"], null_block_id=p["null_block_id"],
                                       chunk_size=p["chunk_size"], seq_order=m["seq_order"])
            da = self.ssd.decode_args(d["x"], d["dt"], d["A"], d["B"], d["C"], d["cache"], self.si_dev, yd,
                                      D=d["D"], dt_bias=d["dt_bias"], null_block_id=d["null_block_id"])
            self.ssd.ssd_mixed_step(pa, da, workspace=self.workspace)
        else:
            if ev is not None:
                ev[0].record()
            self.ssd.ssd_prefill_varlen(p["x"], p["dt"], p["A"], p["B"], p["C"], self.cu_dev,
                                        m["cu_chunk_seqlens"], m["seq_idx"], m["last_chunk_indices"], out=y,
                                        init_slot=m["init_slot"], chunk_slot=m["chunk_slot"],
                                        state_cache=p["cache"], D=p["D"], dt_bias=p["dt_bias"],
                                        null_block_id=p["null_block_id"], chunk_size=p["chunk_size"],
                                        workspace=self.workspace, seq_order=m["seq_order"],
                                        mark=None if ev is None else ev[1])
            if ev is not None:
                ev[2].record()
            if self.dec["live"] > 0:
                self.ssd.ssm_decode_update(d["x"], d["dt"], d["A"], d["B"], d["C"], d["cache"], self.si_dev, None,
                                           out=yd, D=d["D"], dt_bias=d["dt_bias"],
                                           null_block_id=d["null_block_id"])
        if ev is not None:
            ev[3].record()
        if host is not None:
            host["y"].copy_(y, non_blocking=True)
            host["yd"].copy_(yd, non_blocking=True)

    def e2e_pipelined(self, host, steps, mixed):
        """End to end, steps overlapped: step k's inputs go up and step k-1's outputs come down
        while a step computes, on copy streams of their own, with two device buffer sets.  Every
        step still moves its full inputs from pinned host memory and its y back.  Returns the
        device time of all the steps (ms), measured from an event before the first upload to one
        after the last download."""
        comp = torch.cuda.current_stream()
        up, down = torch.cuda.Stream(device=self.dev), torch.cuda.Stream(device=self.dev)
        sets = []
        for _ in range(2):
            b = {}
            for name in ("x", "dt", "B", "C"):
                b["p_" + name] = torch.empty_like(self.pre[name])
                b["d_" + name] = torch.empty_like(self.dec[name])
            b["y"], b["yd"] = torch.empty_like(self.y), torch.empty_like(self.yd)
            sets.append(b)
        ev = lambda: torch.cuda.Event(enable_timing=False)
        landed, used, drained = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(comp)
        up.wait_event(t0)
        for k in range(steps):
            i, b = k % 2, sets[k % 2]
            if k >= 2:
                up.wait_event(used[i])  # step k-2 has finished reading this set
            with torch.cuda.stream(up):
                for name in ("x", "dt", "B", "C"):
                    b["p_" + name].copy_(host["p_" + name], non_blocking=True)
                    b["d_" + name].copy_(host["d_" + name], non_blocking=True)
                landed[i].record(up)
            comp.wait_event(landed[i])
            if k >= 2:
                comp.wait_event(drained[i])  # step k-2's y has reached the host
            self.run(mixed=mixed, bufs=b)
            used[i].record(comp)
            down.wait_event(used[i])
            with torch.cuda.stream(down):
                host["y"].copy_(b["y"], non_blocking=True)
                host["yd"].copy_(b["yd"], non_blocking=True)
                drained[i].record(down)
        comp.wait_stream(up)
        comp.wait_stream(down)
        t1.record(comp)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    def host_buffers(self):
        p, d = self.pre, self.dec
        h = {}
        for name in ("x", "dt", "B", "C"):
            h["p_" + name] = torch.empty(p[name].shape, dtype=p[name].dtype, pin_memory=True)
            h["p_" + name].copy_(p[name])
            h["d_" + name] = torch.empty(d[name].shape, dtype=d[name].dtype, pin_memory=True)
            h["d_" + name].copy_(d[name])
        h["y"] = torch.empty(self.y.shape, dtype=self.y.dtype, pin_memory=True)
        h["yd"] = torch.empty(self.yd.shape, dtype=self.yd.dtype, pin_memory=True)
        h2d = sum(v.numel() * v.element_size() for k, v in h.items() if k[:2] in ("p_", "d_"))
        meta_bytes = sum(v.nbytes for v in self.meta.values())
        d2h = h["y"].numel() * 2 + h["yd"].numel() * 2
        return h, h2d + meta_bytes, d2h


def conv1d_leg(st, steps, warmup):
    """The depthwise causal conv1d in front of the SSM (a next-row step, timed on its own, not
    part of the step above) on the same prefill batch: xBC [T, H*P + 2*G*N] bf16 in, x/B/C out,
    W = 4, conv states read at sequence starts and stored at every chunk end, as the SSM
    states are.  Returns its line object."""
    ssd = st.ssd
    p = st.pre
    T = int(p["cu_seqlens"][-1])
    dim_x, dim_bc, W = st.H * st.P, st.G * st.N, 4
    D = dim_x + 2 * dim_bc
    g = torch.Generator(device=st.dev).manual_seed(11)
    xbc = torch.randn(T, D, generator=g, device=st.dev).to(torch.bfloat16)
    weight = 0.5 * torch.randn(D, W, generator=g, device=st.dev)
    bias = 0.3 * torch.randn(D, generator=g, device=st.dev)
    slots = p["cache"].shape[0]
    state = torch.zeros(slots, W - 1, D, dtype=torch.bfloat16, device=st.dev)
    m = st.device_meta(st.meta)
    S = p["cu_seqlens"].numel() - 1
    outs = st.ssd._binding._conv_outputs(xbc, dim_x, dim_bc, None, None, None)

    def call():
        ssd.ssd_conv1d_varlen(xbc, weight, st.cu_dev, dim_x, dim_bc, bias=bias, conv_state=state,
                              init_slot=m["init_slot"][:S], chunk_slot=m["chunk_slot"][:st.K],
                              cu_chunk_seqlens=m["cu_chunk_seqlens"], last_chunk_indices=m["last_chunk_indices"][:S],
                              null_block_id=p["null_block_id"], x_out=outs[0], B_out=outs[1], C_out=outs[2])
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    nbytes = 2 * T * D * 2 + st.K * (W - 1) * D * 2 + S * (W - 1) * D * 2 + D * (W + 1) * 4
    hbm, _ = _peaks()
    # the decode form on the step's single-token requests: each continues the conv state in its slot
    R = st.dec["live"]
    dec = None
    if R > 0:
        xd = torch.randn(R, D, generator=g, device=st.dev).to(torch.bfloat16)
        si = st.si_dev[:, 0].contiguous()
        douts = st.ssd._binding._conv_outputs(xd, dim_x, dim_bc, None, None, None)

        def dcall():
            ssd.ssd_conv1d_update(xd, weight, state, si, dim_x, dim_bc, bias=bias, null_block_id=p["null_block_id"],
                                  x_out=douts[0], B_out=douts[1], C_out=douts[2])
        dms = _flushed_ms(st.dev, dcall)
        dbytes = 2 * R * D * 2 + 2 * R * (W - 1) * D * 2 + D * (W + 1) * 4
        dec = {"requests": R, "ms_l2_flushed": dms, "algorithmic_bytes": dbytes,
               "hbm_frac_l2_flushed": dbytes / (dms * 1e-3) / 1e9 / hbm}
    return {"what": "depthwise causal conv1d, W=4, silu, %d channels (x %d, B and C %d each)" % (D, dim_x, dim_bc),
            "ms": ms, "tokens_per_s": T / (ms * 1e-3), "algorithmic_bytes": nbytes,
            "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm, "kernels": 2, "decode": dec}


MAMBA1_SHAPE = dict(num_seqs=8, seq_len=8192, dim=5120, dstate=16, ngroups=1, chunk_size=2048, decodes=256)
# The Mamba1 scan is bound by the multi-function unit (one base-2 exponential per token, channel and
# state): 16 results per clock per SM, at the GB300's maximum SM clock.
MUFU_EX2_PER_SM_CLOCK = 16


def mamba1_leg(dev, steps, warmup):
    """The Mamba1 selective scan (a next-row step, timed on its own): 8 fresh sequences of 8192
    tokens, 5120 channels, dstate 16, one group, bf16, states stored at every 2048-token chunk
    end (Mamba1's default chunk); and one decode step of 256 single-token requests on a
    [512, 5120, 16] fp32 cache.  Returns its line object."""
    import selective_state_space_mamba2_gb300 as ssd
    from selective_state_space_mamba2_gb300 import workloads as W
    m = MAMBA1_SHAPE
    S, L, Dc, N, G, Q = m["num_seqs"], m["seq_len"], m["dim"], m["dstate"], m["ngroups"], m["chunk_size"]
    c = W.mamba1_prefill_case(4, [L] * S, [0] * S, Dc, N, G, Q, device=dev, num_slots=S * (L // Q) + 1)
    meta = ssd.ssd_chunk_metadata(c["cu_seqlens"], Q, c["num_computed"], c["has_init"],
                                  block_table=c["block_table"], null_block_id=0)
    K = int(meta["cu_chunk_seqlens"].shape[0] - 1)
    md = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in meta.items()}
    cu = c["cu_seqlens"].to(dev)
    y = torch.empty_like(c["x"])

    def scan():
        ssd.mamba1_scan_varlen(c["x"], c["dt"], c["A"], c["B"], c["C"], cu, md["cu_chunk_seqlens"],
                               md["last_chunk_indices"][:S], D=c["D"], dt_bias=c["dt_bias"], state_cache=c["cache"],
                               init_slot=md["init_slot"][:S], chunk_slot=md["chunk_slot"][:K], out=y)

    R = m["decodes"]
    dc = W.mamba1_decode_case(5, R, R, 1, Dc, N, G, 2 * R + 1, device=dev)
    si = dc["state_indices"].to(dev)
    yd = torch.empty_like(dc["x"])

    def update():
        ssd.mamba1_state_update(dc["x"], dc["dt"], dc["A"], dc["B"], dc["C"], dc["cache"], si, out=yd, D=dc["D"],
                                dt_bias=dc["dt_bias"])

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    # the decode's states (R x Dc x N fp32, read and written in place) fit in L2: it is timed with
    # L2 flushed before every call
    ms, dms = timed(scan), _flushed_ms(dev, update)
    T = S * L
    hbm, _ = _peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = _sm_max_mhz()
    mufu_peak = sms * MUFU_EX2_PER_SM_CLOCK * mhz * 1e6 / 1e12
    nbytes = 3 * T * Dc * 2 + 2 * T * G * N * 2 + K * Dc * N * 4
    dbytes = R * (2 * Dc * N * 4 + 3 * Dc * 2 + 2 * G * N * 2)
    return {"what": "Mamba1 selective scan: %d x %d tokens, %d channels, dstate %d, bf16, states every %d tokens"
                    % (S, L, Dc, N, Q),
            "ms": ms, "tokens_per_s": T / (ms * 1e-3), "algorithmic_bytes": nbytes,
            "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm,
            "exps_per_s": T * Dc * N / (ms * 1e-3),
            "roofline": {"bound": "alu", "achieved": T * Dc * N / (ms * 1e-3) / 1e12, "peak": mufu_peak,
                         "unit": "Tex2/s", "frac": T * Dc * N / (ms * 1e-3) / 1e12 / mufu_peak,
                         "peak_source": "derived: %d SMs x %d ex2 per clock x %.0f MHz"
                                        % (sms, MUFU_EX2_PER_SM_CLOCK, mhz)},
            "decode": {"requests": R, "ms_l2_flushed": dms, "state_updates_per_s": R / (dms * 1e-3),
                       "algorithmic_bytes": dbytes, "hbm_frac_l2_flushed": dbytes / (dms * 1e-3) / 1e9 / hbm},
            "kernels": 2}


# ------------------------------------------------------- the other configs --

L2_FLUSH_BYTES = 512 << 20  # written between repetitions where a config's data fits in the 129 MB L2
SPIN_CYCLES = 20_000_000  # about 10 ms of device spin ahead of a timed loop (the host queues the loop meanwhile)


def _graph_ms(dev, call, per_graph=20, min_s=0.4):
    """Per-call device time of ``call`` replayed back to back: ``per_graph`` calls captured in one
    CUDA graph (so host work between calls cannot leave the GPU idle), the graph replayed until
    ``min_s`` seconds of device time have passed, CUDA events around the replays."""
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            call()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    reps = max(1, int(min_s * 1e3 / max(e0.elapsed_time(e1), 1e-3)))
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * per_graph)


def _flushed_ms(dev, call, reps=40):
    """Median device time of one call with L2 flushed before it: each call sits between CUDA events,
    after a write of L2_FLUSH_BYTES and then a read of another buffer of that size.  The write
    evicts the call's data; the read evicts the write's dirty lines, so their write-back to HBM is
    not charged to the timed call.  A spin kernel first lets the host queue every repetition, so
    the device never waits on the host inside a timed pair."""
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    evict = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda._sleep(200_000_000)
    for a, b in evs:
        flush.fill_(1.0)
        evict.sum()
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def configs_leg(dev):
    """The other workloads of the path, each on its own: the single-sequence warm-up shape
    (2048 tokens = one chunk, H=48, P=64, N=128, G=4; with and without an initial state; L2 flushed
    and not, since its 31 MB fit in L2), the varlen prefix-cached batch (32 requests, U(64,4096) new
    tokens, U(0,8192) computed, chunk 256, half resuming from a 4096-slot cache) and the
    speculative-decode batch (256 live requests padded to 512, 1+3 tokens, U{0..3} accepted, in place
    on an 8192-slot cache; L2 flushed).  Per config: device ms per call, its algorithmic HBM bytes,
    their fraction of the measured copy bandwidth, and the clocks seen while it ran."""
    import selective_state_space_mamba2_gb300 as ssd
    from selective_state_space_mamba2_gb300 import workloads as W
    hbm, _ = _peaks()
    out = {}

    def prefill_call(c):
        meta = ssd.ssd_chunk_metadata(c["cu_seqlens"], c["chunk_size"], c["num_computed"], c["has_init"],
                                      block_table=c["block_table"], state_indices=c["state_indices"],
                                      null_block_id=c["null_block_id"])
        m = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in meta.items()}
        cu = c["cu_seqlens"].to(dev)
        y = torch.empty_like(c["x"])
        a = ssd.prefill_args(c["x"], c["dt"], c["A"], c["B"], c["C"], cu, m["cu_chunk_seqlens"], m["seq_idx"],
                             m["last_chunk_indices"], y, m["init_slot"], m["chunk_slot"], c["cache"], c["D"],
                             c["dt_bias"], chunk_size=c["chunk_size"], seq_order=m["seq_order"])
        ws = torch.empty(max(ssd.ssd_prefill_workspace_size(a), 1), dtype=torch.uint8, device=dev)
        K = int(meta["cu_chunk_seqlens"].shape[0] - 1)
        inits = int(sum(int(v) != c["null_block_id"] for v in meta["init_slot"]))

        def call():
            ssd.ssd_prefill_varlen(c["x"], c["dt"], c["A"], c["B"], c["C"], cu, m["cu_chunk_seqlens"], m["seq_idx"],
                                   m["last_chunk_indices"], out=y, init_slot=m["init_slot"],
                                   chunk_slot=m["chunk_slot"], state_cache=c["cache"], D=c["D"],
                                   dt_bias=c["dt_bias"], null_block_id=c["null_block_id"],
                                   chunk_size=c["chunk_size"], workspace=ws, seq_order=m["seq_order"])
        return call, K, inits, ssd.ssd_prefill_kernel_count(a)

    def entry(T, nbytes, ms, extra=None):
        d = {"ms": ms, "tokens_per_s_per_layer": T / (ms * 1e-3), "algorithmic_bytes": nbytes,
             "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm}
        d.update(extra or {})
        return d

    warm = {"workload": "single-sequence warm-up shape: 2048 tokens = chunk_size, batch 1, H=48, P=64, N=128, G=4, bf16"}
    for name, with_init in (("no_init", False), ("with_init", True)):
        c = W.warmup_shape_prefill(dev, with_init=with_init)
        H, P, N, G = c["x"].shape[1], c["x"].shape[2], c["B"].shape[2], c["B"].shape[1]
        call, K, inits, nk = prefill_call(c)
        nbytes = prefill_bytes(2048, K, H, P, N, G, 2, init_reads=inits)
        with ClockSampler(dev.index) as clk:
            ms = _graph_ms(dev, call)
            msf = _flushed_ms(dev, call)
        warm[name] = entry(2048, nbytes, ms, {"ms_l2_flushed": msf, "hbm_frac_l2_flushed":
                                              nbytes / (msf * 1e-3) / 1e9 / hbm, "kernels": nk,
                                              "clocks": clk.summary()})
        del c, call
    out["warmup_2048"] = warm

    c = W.varlen_prefix_cached_prefill(dev)
    H, P, N, G = c["x"].shape[1], c["x"].shape[2], c["B"].shape[2], c["B"].shape[1]
    T = int(c["cu_seqlens"][-1])
    call, K, inits, nk = prefill_call(c)
    nbytes = prefill_bytes(T, K, H, P, N, G, 2, init_reads=inits)
    with ClockSampler(dev.index) as clk:
        ms = _graph_ms(dev, call, per_graph=10)
    out["varlen_prefix_cached"] = entry(T, nbytes, ms, {
        "workload": "varlen prefix-cached prefill: 32 requests, new U(64,4096), computed U(0,8192), chunk 256, "
                    "half resuming from a [4096,48,64,128] cache; %d tokens, %d chunks, %d initial states"
                    % (T, K, inits), "kernels": nk, "l2": "inputs larger than L2 (no flush)", "clocks": clk.summary()})
    del c, call

    d = W.spec_decode_batch(dev)
    H, P, N, G = d["x"].shape[1], d["x"].shape[2], d["B"].shape[2], d["B"].shape[1]
    si, na = d["state_indices"].to(dev), d["num_accepted"].to(dev)
    yd = torch.empty_like(d["x"])
    tpr = d["tokens_per_req"]
    writes = int((d["state_indices"][:d["live"], :tpr] != d["null_block_id"]).sum())

    def dcall():
        ssd.ssm_decode_update(d["x"], d["dt"], d["A"], d["B"], d["C"], d["cache"], si, na, out=yd, D=d["D"],
                              dt_bias=d["dt_bias"], null_block_id=d["null_block_id"])
    nbytes = decode_bytes(d["live"], tpr, writes, H, P, N, G, 2)
    with ClockSampler(dev.index) as clk:
        msf = _flushed_ms(dev, dcall)
    ups = d["live"] * tpr
    out["spec_decode"] = {"workload": "speculative decode: 256 live requests padded to 512 (null rows), 1+3 tokens, "
                                      "num_accepted U{0..3}, in place on an [8192,48,64,128] fp32 cache",
                          "ms_l2_flushed": msf, "state_updates_per_s": ups / (msf * 1e-3), "algorithmic_bytes": nbytes,
                          "hbm_frac_l2_flushed": nbytes / (msf * 1e-3) / 1e9 / hbm, "kernels": 1,
                          "clocks": clk.summary()}
    return out


def _barrier(dist_on):
    if dist_on:
        torch.distributed.barrier()


def _reduce_over_ranks(v, dist_on, dev, op):
    if not dist_on:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=op)
    return float(t.item())


def _max_over_ranks(v, dist_on, dev):
    """Slowest rank's value (timings: the job ends when the last rank does)."""
    return _reduce_over_ranks(v, dist_on, dev, torch.distributed.ReduceOp.MAX if dist_on else None)


def _sum_over_ranks(v, dist_on, dev):
    """Total over ranks (units of work every rank processed)."""
    return _reduce_over_ranks(v, dist_on, dev, torch.distributed.ReduceOp.SUM if dist_on else None)


def job_rate(local_units, local_ms, steps, dist_on, dev):
    """Whole-job throughput of independent replicas: the units all ranks
    processed over the slowest rank's time.  Returns (units/s, ms per step)."""
    units = _sum_over_ranks(float(local_units), dist_on, dev)
    ms = _max_over_ranks(float(local_ms), dist_on, dev)
    return units / (ms / steps * 1e-3), ms / steps


def _bind_to_gpu_numa(dev):
    """Run this process on the CPUs of the GPU's own NUMA node, so the pinned host buffers of
    the e2e leg (allocated by this thread) sit next to the GPU's host link.  Returns the node,
    or None where the system does not say."""
    try:
        pr = torch.cuda.get_device_properties(dev)
        bdf = "%04x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        with open("/sys/bus/pci/devices/%s/numa_node" % bdf) as f:
            node = int(f.read().strip())
        if node < 0:
            return None
        with open("/sys/devices/system/node/node%d/cpulist" % node) as f:
            cpus = set()
            for part in f.read().strip().split(","):
                lo, _, hi = part.partition("-")
                cpus.update(range(int(lo), int(hi or lo) + 1))
        if cpus:
            os.sched_setaffinity(0, cpus)
            return node
    except (OSError, ValueError, AttributeError):
        pass
    return None


def gpu_arm(args, rank, world, dist_on):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    numa = _bind_to_gpu_numa(dev)
    import selective_state_space_mamba2_gb300 as ssd
    ssd.build()
    wl = WORKLOADS[args.workload]
    st = Step(dev, wl)
    H, P, N, G = st.H, st.P, st.N, st.G
    T = int(st.pre["cu_seqlens"][-1])
    R = st.dec["live"]
    pre_bytes = prefill_bytes(T, st.K, H, P, N, G, 2)
    dec_bytes = decode_bytes(R, 1, R, H, P, N, G, 2)
    mixed = not args.serial_step
    torch.cuda.set_stream(st.stream)
    for _ in range(args.warmup):
        st.run(mixed=mixed)
        st.run()
    torch.cuda.synchronize()

    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        # the step: prefill and decode together (the headline).  A spin kernel ahead of the first
        # event keeps the device busy while the host queues the steps, so that the timed region
        # holds device work only, as in a serving loop whose host runs ahead of the device.
        _barrier(dist_on)
        torch.cuda.synchronize()
        torch.cuda._sleep(SPIN_CYCLES)
        t0.record()
        for i in range(args.steps):
            st.run(mixed=mixed)
        t1.record()
        torch.cuda.synchronize()
        _barrier(dist_on)
        value, ms_step = job_rate(T + R, t0.elapsed_time(t1), args.steps, dist_on, dev)
        # each call on its own (per-call times, the roofline)
        torch.cuda._sleep(SPIN_CYCLES)
        for i in range(args.steps):
            st.run(ev=evs[i])
        torch.cuda.synchronize()
    pre_ms = [e[0].elapsed_time(e[2]) for e in evs]
    fused_ms = [e[1].elapsed_time(e[2]) for e in evs]
    dec_ms = [e[2].elapsed_time(e[3]) for e in evs]

    # end to end: inputs from pinned host memory, y back to host, every step
    e2e_value, e2e_ms, h2d, d2h = None, None, 0, 0
    if not args.no_e2e:
        host, h2d, d2h = st.host_buffers()
        st.e2e_pipelined(host, 2, mixed)  # warm-up (allocates the second buffer set's blocks)
        _barrier(dist_on)
        e2e_value, e2e_ms = job_rate(T + R, st.e2e_pipelined(host, args.steps, mixed), args.steps, dist_on, dev)

    conv = None if args.no_conv else conv1d_leg(st, args.steps, args.warmup)
    m1 = None if args.no_mamba1 else mamba1_leg(dev, args.steps, args.warmup)
    cfgs = None if args.no_configs else configs_leg(dev)
    if rank != 0:
        return None
    hbm, peak_kind = _peaks()
    bf16, bf16_kind = _bf16_peak()
    pre_flops = prefill_mma_flops(st.meta["cu_chunk_seqlens"], H, P, N)
    method_flops = prefill_method_flops(T, H, P, N, G)
    pre_mean = statistics.mean(pre_ms)
    fused_mean = statistics.mean(fused_ms)
    dec_mean = statistics.mean(dec_ms) if R > 0 else 0.0
    achieved = pre_bytes / (pre_mean * 1e-3) / 1e9
    f_bytes = fused_bytes(T, st.K, H, P, N, G, 2)
    f_achieved = f_bytes / (fused_mean * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded randn tokens, -exp(U(0,2)) A, U(-4,-1) dt_bias)",
        "config": dict(wl, parallelism="dp%d (independent replicas)" % world,
                       step="ssd_mixed_step: prefill on the library's high-priority stream, decode beside it on its "
                       "low-priority one, started once the prefill's prep kernel is done"
                       if mixed else "prefill then decode on one stream", host_numa_node=numa),
        "prefill": {"tokens_per_s_per_layer": T / (pre_mean * 1e-3), "ms": pre_mean,
                    "algorithmic_bytes": pre_bytes,
                    "hbm_frac": achieved / hbm,
                    "what": "the whole call (%d kernels): its algorithmic bytes / its time" % st.prefill_kernels,
                    "fused_kernel_ms": fused_mean, "prep_ms": pre_mean - fused_mean,
                    "tensor": {"achieved": pre_flops / (fused_mean * 1e-3) / 1e12, "peak": bf16,
                               "unit": "TFLOP/s", "frac": pre_flops / (fused_mean * 1e-3) / 1e12 / bf16,
                               "flops": pre_flops, "peak_source": bf16_kind,
                               "what": "tcgen05 flops the fused kernel issues (four products per 128-token "
                                       "block and head on full tiles, fp16 operands, fp32 accumulators) / "
                                       "the fused kernel's time"},
                    "method_flops": {"flops": method_flops,
                                     "achieved": method_flops / (fused_mean * 1e-3) / 1e12, "unit": "TFLOP/s",
                                     "frac": method_flops / (fused_mean * 1e-3) / 1e12 / bf16,
                                     "what": "G Q N + H Q P + 4 H P N per token at Q = 128 (the causal halves "
                                             "only, C B^T once per group) / the fused kernel's time"}},
        "mixed_step": {"ms": ms_step, "prefill_alone_ms": pre_mean, "decode_alone_ms": dec_mean,
                       "serial_ms": pre_mean + dec_mean,
                       "bound_ms": pre_mean,
                       "what": "the step with the decode beside the prefill; bound_ms is the step if the decode "
                               "were hidden entirely (prefill alone), the most a single persistent launch could "
                               "give"},
        "decode": {"state_updates_per_s": R / (dec_mean * 1e-3) if R else None, "ms": dec_mean,
                   "algorithmic_bytes": dec_bytes,
                   "hbm_frac": dec_bytes / (dec_mean * 1e-3) / 1e9 / hbm if R else None},
        "roofline": {"kernel": "ssd_prefill_tc_kernel (the fused kernel of ssd_prefill_varlen)", "bound": "hbm",
                     "achieved": f_achieved, "peak": hbm, "unit": "GB/s", "frac": f_achieved / hbm,
                     "traffic": prefill_traffic(T, H, P, N, G, fused_only=True),
                     "traffic_source": FUSED_TRAFFIC_SOURCE, "peak_source": peak_kind,
                     "algorithmic_bytes": f_bytes, "ms": fused_mean,
                     "units": "the kernel's algorithmic bytes per launch (the call's, less dt, which the prep "
                              "kernel reads) / its mean launch time, CUDA events on its stream: one the library "
                              "records right before the launch (ssd_prefill_varlen_marked), one after the call",
                     "call": {"kernels": st.prefill_kernels, "achieved": achieved, "frac": achieved / hbm,
                              "traffic": prefill_traffic(T, H, P, N, G), "traffic_source": PREFILL_TRAFFIC_SOURCE}},
        "clocks": clk.summary(),
        "e2e": None if e2e_ms is None else {"value": e2e_value, "unit": UNIT,
                                            "how": "every step uploads its inputs from pinned host memory and "
                                                   "downloads y; uploads, compute and downloads of consecutive "
                                                   "steps overlap on three streams (two device buffer sets)",
                                            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": (st.prefill_kernels + (1 if R else 0)) * args.steps,
        "conv1d": conv,
        "mamba1": m1,
        "configs": cfgs,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


# -------------------------------------------------------------- CPU arm -----

def _oracle_sample(tokens, seed=4):
    """A prefix of one prefill sequence of the same workload (all 128 heads),
    generated on the CPU with the workload's distributions."""
    from selective_state_space_mamba2_gb300 import workloads as W
    c = W.prefill_case(seed, [tokens], [0], WORKLOAD["nheads"], WORKLOAD["headdim"], WORKLOAD["dstate"],
                       WORKLOAD["ngroups"], WORKLOAD["chunk_size"], device="cpu", num_slots=2, mode="default")
    return c


def _time_oracle(c, threads):
    import oracle
    T = c["x"].shape[0]
    cc = np.arange(0, T + 1, WORKLOAD["chunk_size"], dtype=np.int32)
    if cc[-1] != T:
        cc = np.append(cc, T).astype(np.int32)
    args = [c[k].double().numpy() for k in ("x", "dt", "A", "B", "C")]
    t = time.perf_counter()
    oracle.ssd_prefill(args[0], args[1], args[2], args[3], args[4], [0, T], cc, D=c["D"], dt_bias=c["dt_bias"],
                       nthreads=threads)
    return time.perf_counter() - t


def cpu_baseline(target_s=15.0):
    import oracle
    threads = oracle.default_threads()
    probe = 256
    dt = _time_oracle(_oracle_sample(probe), threads)
    tokens = int(max(probe, min(65536, probe * target_s / max(dt, 1e-3))))
    tokens = max(256, (tokens // 256) * 256)
    c = _oracle_sample(tokens)
    times = [_time_oracle(c, threads)]
    # one sequence is the largest sample held on the host; repeat it until about target_s of work
    while sum(times) + times[0] <= target_s:
        times.append(_time_oracle(c, threads))
    dt = statistics.mean(times)
    return {"value": tokens / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "first %d tokens of one 65536-token prefill, all 128 heads, fp64 sequential recurrence, "
                      "timed %d times (%.1f s in all)" % (tokens, len(times), sum(times))}


def reference_arm(args, rank):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    probe = 256
    dt = _time_oracle(_oracle_sample(probe), threads)
    budget = 150.0 / max(args.steps + args.warmup, 1)  # whole run within a few minutes
    tokens = max(256, (int(probe * budget / max(dt, 1e-3)) // 256) * 256)
    tokens = min(tokens, 65536)
    c = _oracle_sample(tokens)
    for _ in range(args.warmup):
        _time_oracle(c, threads)
    times = [_time_oracle(c, threads) for _ in range(args.steps)]
    v = tokens / statistics.mean(times)
    return {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": statistics.mean(times) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(WORKLOAD, parallelism="host cores"), "impl": "reference",
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": "first %d tokens of one 65536-token prefill, all 128 heads" % tokens},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--workload", default="long_mixed", choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiler runs)")
    ap.add_argument("--no-conv", action="store_true", help="skip the conv1d measurement")
    ap.add_argument("--no-mamba1", action="store_true", help="skip the Mamba1 measurement")
    ap.add_argument("--no-configs", action="store_true", help="skip the warm-up, varlen and spec-decode configs")
    ap.add_argument("--serial-step", action="store_true", help="run the step's decode after the prefill on one stream")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist_on = world > 1
    if args.impl == "reference":
        line = reference_arm(args, rank)
    else:
        args.warmup = max(args.warmup, 3)  # timing rule: at least 3 warm-up steps
        if dist_on:
            torch.distributed.init_process_group("nccl")
        line = gpu_arm(args, rank, world, dist_on)
        if dist_on:
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
