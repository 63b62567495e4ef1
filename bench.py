#!/usr/bin/env python
"""Benchmark of the GDN layer hot path on GB300.

One step = one Qwen3.5-27B-shaped GDN layer prefill of one 4096-token sequence
(token-major, Hk=16 q/k heads, Hv=48 v heads, dk=dv=128, chunk 64): the width-4 conv1d +
SiLU over the 10240 packed q||k||v channels, then the chunked gated delta rule with
in-kernel q/k L2 norm.  `value` is prefill tokens/s per layer over all ranks.  The decode
half of the metric (256 sequences, one token each, fp32 state [256,48,128,128] updated in
place, conv update over 10240 channels) is timed in the same run and reported under
"decode" in state GB/s against HBM.

Timing: W untimed warm-up steps, then K steps bracketed by barrier + synchronize;
per-kernel CUDA events on the launching stream (torch's current stream); L2 flushed by a
256 MiB write and a 256 MiB read of another buffer between prefill steps (the read drains
the write's dirty lines before the timed region; the decode state, 805 MB, exceeds L2 by
itself);
max over ranks.  `e2e` repeats the prefill through the public API with pinned host
inputs copied in and the outputs (o, final state) read back inside the timed region;
the sequence goes through in four pieces so the copies overlap the layer (each piece
continues the previous one's state; the output is checked equal to the one-call layer's).

--impl reference times the fp64 CPU oracle on the host cores on the same workload
(the reference arm of this project; the pages publish no implementation to run).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "GDN prefill tokens/s per layer (% bf16 TC peak); decode step state GB/s vs HBM"
SHAPE = dict(Hk=16, Hv=48, dk=128, dv=128)
CHUNK = 64
# Pieces of the sequence in the e2e leg's copy / compute pipeline, in sixteenths of T.
# The host link is the bound (all inputs take ~0.41 ms to copy in, the outputs ~0.28 ms
# out), so a small first piece lets the first copy-out start early, the pieces shrink
# toward the end so that little runs after the last copy-in, and there are few pieces,
# each of which costs host time.
E2E_SIXTEENTHS = (2, 7, 5, 2)


def prefill_flops_per_token(Hk, Hv, dk, dv, C=CHUNK):
    """Algorithmic FLOPs per token of the chunked scan (WY/UT form, per chunk of C):
    KK^T and QK^T per k-head (2 x 2*C*dk per token); per v-head the C-sized products
    Tinv*K', Tinv*V', M*Vnew (3 x 2*C*d) and the d-sized products W*S, Q*S, K^T*Vnew
    (3 x 2*d*d); the unit-triangular solve C^2/3 per token per v-head."""
    d = dk
    return Hk * 2 * 2 * C * d + Hv * 2 * (3 * C * d + 3 * d * dv) + Hv * C * C / 3.0


def prefill_bytes(T, N, Hk, Hv, dk, dv, init_state=False):
    act = T * (2 * Hk * dk + 2 * Hv * dv) * 2 + T * Hv * 4 * 2
    st = N * Hv * dk * dv * 4 * (2 if init_state else 1)
    return act + st


def conv_bytes(T, C, N, with_state=False):
    return T * C * 2 * 2 + C * 4 * 2 + (N * 3 * C * 2 * (2 if with_state else 1))


def decode_bytes(N, Hk, Hv, dk, dv, C):
    state = 2 * N * Hv * dk * dv * 4
    act = N * (2 * Hk * dk + 2 * Hv * dv) * 2 + N * Hv * 4 * 2
    conv = N * C * 2 * 2 + 2 * N * 3 * C * 2 + C * 4 * 2
    return state + act + conv, state


def kernel_traffic(src_name):
    """DRAM bytes per launch (read + write) from the last ncu capture of a kernel file, if
    that capture was taken from the current sources, else None.  The record lists the
    files whose device code the kernel compiles from (the .cu file and the headers it
    takes device code from); it holds the sha1 of their contents, concatenated in that
    order."""
    import hashlib
    csrc = os.path.join(ROOT, "gated_deltanet_linear_11_gb300", "csrc")
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(src_name)
        if not rec:
            return None
        h = hashlib.sha1()
        for name in rec.get("sources", [src_name]):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
    except (OSError, ValueError):
        return None
    if rec.get("sha1") != h.hexdigest():
        return None
    return rec.get("dram_bytes_per_launch")


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    out = dict(FALLBACK_PEAKS)
    src = "fallback"
    try:
        with open(path) as f:
            m = json.load(f)

        def find(keys):
            for k in keys:
                if k in m and isinstance(m[k], (int, float)):
                    return float(m[k])
            return None
        hb = find(["hbm_gbs", "hbm_GBps", "hbm_copy_gbs"])
        tf = find(["bf16_tflops", "bf16_dense_tflops"])
        ts = find(["bf16_tflops_sustained"])
        if hb and tf:
            out.update(hbm_gbs=hb, bf16_tflops=tf)
            if ts:
                out["bf16_tflops_sustained"] = ts
            src = "measured"
    except (OSError, ValueError):
        pass
    out["source"] = src
    return out


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "200"], stdout=self.file,
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for nm, val in zip(names, r[5:9]):
                    if val.strip().lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------- our arm

def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import gated_deltanet_linear_11_gb300 as gdn
    from gated_deltanet_linear_11_gb300 import build as gbuild
    from gated_deltanet_linear_11_gb300 import inputs

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    gbuild.build()
    gdn.load()
    peaks = read_peaks()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    launches = 0

    # ---------------- prefill workload (27B layer, one 4096-token sequence)
    T = args.T
    s = SHAPE
    C = inputs.conv_channels(**s)
    wl = inputs.layer_27b(seed=2, T=T)
    cv = wl["conv"]
    x = cv["x"].to(dev)
    w = cv["w"].to(dev)
    g = wl["g"].to(dev)
    beta = wl["beta"].to(dev)
    cu_h = cv["cu_seqlens"]
    cu = cu_h.to(dev)
    y = torch.empty_like(x)
    conv_out = torch.empty((1, 3, C), dtype=torch.bfloat16, device=dev)
    o = torch.empty((T, s["Hv"], s["dv"]), dtype=torch.bfloat16, device=dev)
    hT = torch.empty((1, s["Hv"], s["dk"], s["dv"]), dtype=torch.float32, device=dev)
    ws_bytes = gdn.gdn_chunk_prefill_workspace_size(1, T, s["Hk"], s["Hv"], 128, 128, CHUNK)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    # L2 flush between steps: a 256 MiB write, then a 256 MiB read of another buffer, which
    # evicts the written (dirty) lines so their write-back happens before the timed region
    # rather than under the first kernel of the step
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.int32, device=dev)
    flush_rd = torch.zeros(64 * 1024 * 1024, dtype=torch.int32, device=dev)

    def flush_l2():
        flush.zero_()
        flush_rd.max()
    q_v, k_v, v_v = gdn.split_qkv(y, s["Hk"], s["Hv"], s["dk"], s["dv"])
    # the layer entry runs the v channels' conv on this second stream, under the chunk
    # preparation
    side = torch.cuda.Stream(device=dev)

    scan_launches = 2 if ws_bytes else 1   # tensor-core path: prep + state kernels
    legs = set(args.legs.split(","))
    clk, t_wall, ms_step, value = None, None, None, None
    scan_avg = conv_avg = achieved_tf = None
    flops = prefill_flops_per_token(**s) * T
    conv_b = conv_bytes(T, C, 1)
    scan_b = prefill_bytes(T, 1, **s)

    if "prefill" in legs:
        # (1) the step: one gdn_layer_prefill call (conv over q|k|v, then the chunk scan;
        #     the v channels' conv runs on the caller's side stream under the chunk
        #     preparation), timed as a whole; also timed with the v channels' conv fused
        #     into the state pass (GDN_LAYER_FUSED_VCONV), for the record
        def layer_step(fused=False):
            gdn.gdn_layer_prefill(x, w, None, g, beta, cu, s["Hk"], s["Hv"], s["dk"], s["dv"],
                                  conv_state_out=conv_out, o=o, final_state=hT, y=y,
                                  cu_seqlens_host=cu_h, workspace=ws,
                                  side_stream=None if fused else side, fused_vconv=fused)

        # (2) the same work as two calls, each bracketed, for the per-kernel roofline
        def component_step(evs):
            evs[0].record(stream)
            gdn.gdn_conv1d_fwd(x, w, None, cu, None, conv_out, y, cu_seqlens_host=cu_h)
            evs[1].record(stream)
            gdn.gdn_chunk_prefill(q_v, k_v, v_v, g, beta, cu, chunk=CHUNK, l2norm=True,
                                  o=o, final_state=hT, cu_seqlens_host=cu_h, workspace=ws)
            evs[2].record(stream)

        for _ in range(args.warmup):
            flush_l2()
            layer_step()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        clocks = Clocks(local).start()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush_l2()
            sevs[i][0].record(stream)
            layer_step()
            sevs[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        barrier(world)
        clk = clocks.stop()
        step_ms = [e[0].elapsed_time(e[1]) for e in sevs]
        launches += args.steps * (2 + scan_launches)
        ms_step = max_over_ranks(statistics.mean(step_ms), world)
        value = world * T / (ms_step * 1e-3)

        for _ in range(args.warmup):
            flush_l2()
            layer_step(True)
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush_l2()
            sevs[i][0].record(stream)
            layer_step(True)
            sevs[i][1].record(stream)
        torch.cuda.synchronize()
        launches += args.steps * (1 + scan_launches)
        vconv_fused_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in sevs)

        for _ in range(args.warmup):
            flush_l2()
            component_step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2()
            component_step(evs[i])
        torch.cuda.synchronize()
        launches += args.steps * (1 + scan_launches)
        conv_ms = [e[0].elapsed_time(e[1]) for e in evs]
        scan_ms = [e[1].elapsed_time(e[2]) for e in evs]
        scan_avg = statistics.mean(scan_ms)
        conv_avg = statistics.mean(conv_ms)

        # the conv at 6144 channels, the workloads' literal "6144-wide packed qkv" reading
        # (Hv*dv alone), reported beside the 10240-channel q|k|v conv the layer runs
        C6 = s["Hv"] * s["dv"]
        x6 = torch.empty((T, C6), dtype=torch.bfloat16, device=dev).copy_(x[:, 2 * s["Hk"] * s["dk"]:])
        w6 = w[2 * s["Hk"] * s["dk"]:].contiguous()
        y6 = torch.empty_like(x6)
        cs6 = torch.empty((1, 3, C6), dtype=torch.bfloat16, device=dev)
        for _ in range(args.warmup):
            flush_l2()
            gdn.gdn_conv1d_fwd(x6, w6, None, cu, None, cs6, y6, cu_seqlens_host=cu_h)
        torch.cuda.synchronize()
        c6_ms = []
        for i in range(args.steps):
            flush_l2()
            evs[i][0].record(stream)
            gdn.gdn_conv1d_fwd(x6, w6, None, cu, None, cs6, y6, cu_seqlens_host=cu_h)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        launches += args.steps
        conv6_avg = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
        conv6_b = conv_bytes(T, C6, 1)
        del x6, y6

        achieved_tf = flops / (scan_avg * 1e-3) / 1e12

    decode = None
    if "decode" in legs:
        # ---------------- decode workload (256 sequences, fp32 state pool 805 MB)
        Nd = args.decode_n
        dd = inputs.decode_27b(seed=4, N=Nd)
        dx = dd["conv"]["x"].to(dev)
        dcs = dd["conv"]["conv_state"].to(dev)
        dw = torch.empty((C, 4), dtype=torch.bfloat16, device=dev).copy_(cv["w"])
        dq, dk_, dvv = dd["q"].to(dev), dd["k"].to(dev), dd["v"].to(dev)
        dg, db = dd["g"].to(dev), dd["beta"].to(dev)
        pool = dd["state_pool"].to(dev)
        idx = dd["state_idx"].to(dev)
        dy = torch.empty_like(dx)
        do = torch.empty((Nd, s["Hv"], s["dv"]), dtype=torch.bfloat16, device=dev)
        dstatus = torch.zeros(1, dtype=torch.int32, device=dev)

        def decode_step(evs=None):
            if evs:
                evs[0].record(stream)
            gdn.gdn_conv1d_update(dx, dw, None, dcs, idx, dy, dstatus)
            if evs:
                evs[1].record(stream)
            gdn.gdn_recurrent_decode(dq, dk_, dvv, dg, db, pool, idx, 1.0, True, do, dstatus)
            if evs:
                evs[2].record(stream)

        for _ in range(args.warmup):
            decode_step()
        torch.cuda.synchronize()
        barrier(world)
        devs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for i in range(args.steps):
            decode_step(devs[i])
        torch.cuda.synchronize()
        barrier(world)
        launches += 2 * args.steps
        dconv_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in devs)
        ddec_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in devs)
        dstep_ms = max_over_ranks(dconv_ms + ddec_ms, world)
        dbytes, dstate = decode_bytes(Nd, s["Hk"], s["Hv"], s["dk"], s["dv"], C)
        dconv_b = Nd * C * 2 * 2 + 2 * Nd * 3 * C * 2
        dec_b = dbytes - dconv_b
        assert int(dstatus.item()) == 0
        decode = {"workload": "%d seqs x 1 token, state [%d,48,128,128] fp32 in place, "
                              "conv update 10240 ch, permuted state_idx" % (Nd, Nd),
                  "ms_per_step": dstep_ms,
                  "state_gbs": dstate / (dstep_ms * 1e-3) / 1e9,
                  "kernels_ms": {"conv1d_update": dconv_ms, "recurrent_decode": ddec_ms},
                  "roofline": {"kernel": "recurrent_decode", "bound": "hbm",
                               "achieved": dec_b / (ddec_ms * 1e-3) / 1e9,
                               "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": dec_b / (ddec_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                               "traffic": kernel_traffic("decode.cu")}}

        # the conv update over 6144 channels too (the literal "6144-wide" reading)
        cv0 = 2 * s["Hk"] * s["dk"]
        dx6 = dx[:, cv0:].contiguous()
        dw6 = dw[cv0:].contiguous()
        dcs6 = dcs[:, :, cv0:].contiguous()
        dy6 = torch.empty_like(dx6)
        # (each launch after an L2 flush, which also keeps the GPU busy while the host
        # enqueues the next launch, so that no launch gap is timed)
        for _ in range(args.warmup):
            flush_l2()
            gdn.gdn_conv1d_update(dx6, dw6, None, dcs6, idx, dy6, dstatus)
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush_l2()
            devs[i][0].record(stream)
            gdn.gdn_conv1d_update(dx6, dw6, None, dcs6, idx, dy6, dstatus)
            devs[i][1].record(stream)
        torch.cuda.synchronize()
        launches += args.steps
        d6_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in devs)
        C6 = dx6.shape[1]
        d6_b = Nd * C6 * 2 * 2 + 2 * Nd * 3 * C6 * 2
        decode["conv_update_literal_6144"] = {
            "ms": d6_ms, "achieved": d6_b / (d6_ms * 1e-3) / 1e9, "unit": "GB/s",
            "frac": d6_b / (d6_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        del dx6, dcs6, dy6

        # ---------------- the same step in one launch: gdn_fused_decode from gate logits
        grng = np.random.default_rng(7)
        a_raw = torch.from_numpy(grng.standard_normal((Nd, s["Hv"])) + 2.0).float().to(dev)
        b_raw = torch.from_numpy(grng.standard_normal((Nd, s["Hv"]))).float().to(dev)
        dx_c = dx.contiguous()

        def fused_step():
            gdn.gdn_fused_decode(dx_c, dw, None, a_raw, b_raw, dcs, pool, s["Hk"], s["Hv"],
                                 s["dk"], s["dv"], state_idx=idx, l2norm=True, o=do,
                                 status=dstatus)

        for _ in range(args.warmup):
            fused_step()
        torch.cuda.synchronize()
        barrier(world)
        fevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            fevs[i][0].record(stream)
            fused_step()
            fevs[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        launches += 2 * args.steps
        fused_ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in fevs), world)
        assert int(dstatus.item()) == 0
        decode["fused"] = {"kernel": "fused_decode (conv update + gates + recurrent step)",
                           "ms_per_step": fused_ms,
                           "state_gbs": dstate / (fused_ms * 1e-3) / 1e9,
                           "roofline": {"bound": "hbm",
                                        "achieved": dbytes / (fused_ms * 1e-3) / 1e9,
                                        "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                        "frac": dbytes / (fused_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}}

    e2e = None
    o_ref = o.clone() if "prefill" in legs else None   # the unsplit layer's output
    if "e2e" in legs:
        # ---------------- e2e: pinned host inputs in, outputs out, through the public API
        hx = cv["x"].pin_memory()
        hg = wl["g"].pin_memory()
        hb = wl["beta"].pin_memory()
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hh = torch.empty(hT.shape, dtype=hT.dtype).pin_memory()
        e2e_steps = max(3, min(args.steps, 10))
        # The sequence is fed in pieces (multiples of the 64-token chunk): piece i+1 is
        # copied in while piece i runs, and piece i's output is copied out while piece i+1
        # runs.  Each piece continues from the previous one's recurrent state and conv
        # state, which reproduces the unsplit call bit for bit.
        if T % (64 * 16) == 0:
            plens = [T * k // 16 for k in E2E_SIXTEENTHS]
        else:
            plens = [T]
        parts = len(plens)
        bounds = [sum(plens[:i]) for i in range(parts + 1)]
        h2d_stream = torch.cuda.Stream(device=dev)
        d2h_stream = torch.cuda.Stream(device=dev)
        part_cu = [torch.tensor([0, n], dtype=torch.int32) for n in plens]
        part_cu_d = [c.to(dev) for c in part_cu]
        conv_states = [torch.empty_like(conv_out), torch.empty_like(conv_out)]

        def e2e_step():
            start = torch.cuda.Event()
            start.record(stream)
            h2d_stream.wait_event(start)
            d2h_stream.wait_event(start)
            for i in range(parts):
                a, b = bounds[i], bounds[i + 1]
                with torch.cuda.stream(h2d_stream):
                    x[a:b].copy_(hx[a:b], non_blocking=True)
                    g[a:b].copy_(hg[a:b], non_blocking=True)
                    beta[a:b].copy_(hb[a:b], non_blocking=True)
                    arrived = torch.cuda.Event()
                    arrived.record(h2d_stream)
                stream.wait_event(arrived)
                gdn.gdn_layer_prefill(x[a:b], w, None, g[a:b], beta[a:b], part_cu_d[i], s["Hk"],
                                      s["Hv"], s["dk"], s["dv"],
                                      conv_state_in=None if i == 0 else conv_states[(i - 1) & 1],
                                      conv_state_out=conv_states[i & 1],
                                      initial_state=None if i == 0 else hT, final_state=hT,
                                      y=y[a:b], o=o[a:b], cu_seqlens_host=part_cu[i],
                                      workspace=ws, side_stream=side)
                computed = torch.cuda.Event()
                computed.record(stream)
                d2h_stream.wait_event(computed)
                with torch.cuda.stream(d2h_stream):
                    ho[a:b].copy_(o[a:b], non_blocking=True)
            with torch.cuda.stream(d2h_stream):
                hh.copy_(hT, non_blocking=True)
            finished = torch.cuda.Event()
            finished.record(d2h_stream)
            stream.wait_event(finished)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        launches += e2e_steps * parts * (2 + scan_launches)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
        if o_ref is not None:
            # the pieces continue each other exactly: same bits as the one-call layer
            assert torch.equal(ho, o_ref.cpu()), "pipelined e2e output differs from the layer's"

        h2d = hx.numel() * 2 + hg.numel() * 4 + hb.numel() * 4
        d2h = ho.numel() * 2 + hh.numel() * 4
        e2e = {"value": world * T / (e2e_ms * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "pipeline": "%d pieces of %s tokens: copy-in, layer and copy-out overlap"
                            % (parts, "+".join(str(n) for n in plens))}

    result = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 (fp32 state and accumulation)",
        "data": "synthetic (seeded; Qwen3.5-27B head shapes, random conv weights)",
        "config": {"workload": "qwen3.5-27b GDN layer prefill, 1 seq x %d tokens, Hk=16 "
                               "Hv=48 dk=dv=128, conv 10240 ch, chunk 64, q/k L2 norm "
                               "in kernel" % T,
                   "global_batch": world, "seq_len": T, "parallelism": "replicas x%d" % world,
                   "l2": "flushed between steps (256 MiB write, then a 256 MiB read)"},
    }
    if "prefill" in legs:
        result["kernels_ms"] = {"conv1d_fwd": conv_avg, "chunk_prefill": scan_avg,
                                "conv_plus_chunk_as_two_calls": conv_avg + scan_avg,
                                "layer_v_conv_fused_into_state_pass": vconv_fused_ms}
        result["roofline"] = {
            "kernel": "chunk_prefill", "bound": "tensor", "achieved": achieved_tf,
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved_tf / peaks["bf16_tflops"],
            "peak_source": "%s (bf16 dense burst)" % peaks["source"],
            "traffic": kernel_traffic("chunk_tc.cu"),
            "traffic_note": "dram bytes of prep + state kernels per launch pair (ncu)",
            "algorithmic_flops_per_launch": flops,
            "algorithmic_bytes_per_launch": scan_b,
            "hbm_gbs_equiv": scan_b / (scan_avg * 1e-3) / 1e9}
        result["conv_roofline"] = {
            "bound": "hbm", "achieved": conv_b / (conv_avg * 1e-3) / 1e9,
            "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": conv_b / (conv_avg * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "traffic": kernel_traffic("conv1d.cu")}
        result["conv_literal_6144"] = {
            "workload": "conv1d_fwd over [%d, %d] (the literal 6144-wide reading)" % (T, C6),
            "ms": conv6_avg, "achieved": conv6_b / (conv6_avg * 1e-3) / 1e9,
            "unit": "GB/s", "frac": conv6_b / (conv6_avg * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        result["clocks"] = clk
        result["wall_s_timed_region"] = t_wall
    if decode is not None:
        result["decode"] = decode
    if e2e is not None:
        result["e2e"] = e2e
    if "multiseq" in legs:
        multiseq, n = multiseq_leg(gdn, inputs, dev, flush_l2, peaks["bf16_tflops"],
                                   args.warmup, min(args.steps, 10))
        result["multiseq"] = multiseq
        launches += n
    result["gpu_launches"] = launches
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(T, samples=args.cpu_samples)
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# -------------------------------------------------------------- oracle on the host

def oracle_layer_once(T, v_heads=None):
    import oracle
    from gated_deltanet_linear_11_gb300 import inputs
    wl = inputs.layer_27b(seed=2, T=T)
    cv = wl["conv"]
    t0 = time.perf_counter()
    oracle.layer_prefill(cv["x"], cv["w"], None, wl["g"], wl["beta"], cv["cu_seqlens"],
                         v_heads=v_heads, **SHAPE)
    return time.perf_counter() - t0


def cpu_baseline(T, samples=3):
    import oracle
    oracle.build()
    times = [oracle_layer_once(T) for _ in range(samples)]
    t = statistics.median(times)
    return {"value": T / t, "unit": "tokens/s", "cores": oracle.default_threads(),
            "kind": "oracle",
            "sample": "fp64 oracle layer prefill (conv + token recurrence), the full "
                      "%d-token 27B-shaped workload, median of %d runs" % (T, samples)}


def multiseq_leg(gdn, inputs, dev, flush_l2, peak_tf, warmup, steps):
    """The chunk scan alone on packed multi-sequence batches.  Inputs are
    drawn on the device from a seeded generator with the workloads' distributions: unit
    q/k rows, v ~ N(0,1), g = -softplus(N(0,1) + 2), beta = sigmoid(N(0,1)), initial
    states ~ N(0, 0.02) where the workload continues sequences.  Returns one record per
    workload and the number of kernel launches."""
    import torch
    fresh, cont, _ = inputs.mix_lengths(5)
    cases = [("27B shapes, 8 x 4096 tokens", [4096] * 8, 16, 48, False),
             ("27B shapes, 8 sequences U[1, 8192], initial states",
              inputs.varlen_lengths(3), 16, 48, True),
             ("4B shapes, the mix's 40 prefills: 20 fresh U[12, 32768] and 20 continuations "
              "of 2048 on initial states", fresh + cont, 16, 32, True)]
    # a head-sharded layer (the 27B heads over 8 GPUs of tensor parallelism: Hk=2, Hv=6)
    # on one long sequence: its 18 chains leave most SMs idle, so the scan also runs
    # context-parallel, in ranges of 32 and of 64 chunks (range_chunks, last field)
    cases += [("27B heads / 8 (Hk=2, Hv=6), 1 x 32768 tokens", [32768], 2, 6, True, 0),
              ("27B heads / 8 (Hk=2, Hv=6), 1 x 32768 tokens, context-parallel in ranges "
               "of 64 chunks", [32768], 2, 6, True, 64),
              ("27B heads / 8 (Hk=2, Hv=6), 1 x 32768 tokens, context-parallel in ranges "
               "of 32 chunks", [32768], 2, 6, True, 32)]
    # and in the range length gdn_chunk_prefill_cp_range_hint picks for that sequence
    hint = gdn.gdn_chunk_prefill_cp_range_hint(32768, 6)
    if hint:
        cases.append(("27B heads / 8 (Hk=2, Hv=6), 1 x 32768 tokens, context-parallel in "
                      "ranges of %d chunks (the range hint)" % hint, [32768], 2, 6, True, hint))
    cases = [c if len(c) == 6 else c + (0,) for c in cases]
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    out, launches = [], 0
    for name, lens, Hk, Hv, init, range_chunks in cases:
        T, N = sum(lens), len(lens)

        def unit_rows(t):
            return (t / t.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
        q = unit_rows(torch.randn(T, Hk, 128, device=dev, generator=gen))
        k = unit_rows(torch.randn(T, Hk, 128, device=dev, generator=gen))
        v = torch.randn(T, Hv, 128, device=dev, generator=gen).to(torch.bfloat16)
        g = -torch.nn.functional.softplus(torch.randn(T, Hv, device=dev, generator=gen) + 2)
        beta = torch.sigmoid(torch.randn(T, Hv, device=dev, generator=gen))
        cu_h = torch.zeros(N + 1, dtype=torch.int32)
        cu_h[1:] = torch.cumsum(torch.tensor(lens), 0)
        cu = cu_h.to(dev)
        h0 = torch.randn(N, Hv, 128, 128, device=dev, generator=gen) * 0.02 if init else None
        o = torch.empty((T, Hv, 128), dtype=torch.bfloat16, device=dev)
        hT = torch.empty((N, Hv, 128, 128), dtype=torch.float32, device=dev)
        if range_chunks:
            ws_bytes = gdn.gdn_chunk_prefill_cp_workspace_size(cu_h, T, Hk, Hv, 128, 128,
                                                               range_chunks, CHUNK)
        else:
            ws_bytes = gdn.gdn_chunk_prefill_workspace_size(N, T, Hk, Hv, 128, 128, CHUNK)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)

        def scan():
            if range_chunks:
                gdn.gdn_chunk_prefill_cp(q, k, v, g, beta, cu, range_chunks, chunk=CHUNK,
                                         initial_state=h0, o=o, final_state=hT,
                                         cu_seqlens_host=cu_h, workspace=ws)
            else:
                gdn.gdn_chunk_prefill(q, k, v, g, beta, cu, chunk=CHUNK, initial_state=h0,
                                      o=o, final_state=hT, cu_seqlens_host=cu_h,
                                      workspace=ws)
        for _ in range(warmup):
            flush_l2()
            scan()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for e0, e1 in evs:
            flush_l2()
            e0.record()
            scan()
            e1.record()
        torch.cuda.synchronize()
        launches += (5 if range_chunks else 2) * steps
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        tf = prefill_flops_per_token(Hk, Hv, 128, 128) * T / (ms * 1e-3) / 1e12
        out.append({"workload": name, "tokens": T, "sequences": N, "longest": max(lens),
                    "range_chunks": range_chunks or None,
                    "ms": ms, "tokens_per_s": T / (ms * 1e-3), "tflops": tf,
                    "frac": tf / peak_tf,
                    "roofline": {"kernel": "chunk_prefill", "bound": "tensor", "achieved": tf,
                                 "peak": peak_tf, "unit": "TFLOP/s", "frac": tf / peak_tf,
                                 "traffic": None}})
        del q, k, v, g, beta, o, hT, ws, h0
        torch.cuda.empty_cache()
    return out, launches


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    T = args.T
    for _ in range(args.warmup):
        oracle_layer_once(T)
    times = [oracle_layer_once(T) for _ in range(args.steps)]
    t = statistics.mean(times)
    value = T / t
    cores = oracle.default_threads()
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": "qwen3.5-27b GDN layer prefill, 1 seq x %d tokens, Hk=16 "
                                  "Hv=48 dk=dv=128, conv 10240 ch, chunk 64, q/k L2 norm "
                                  "in kernel" % T, "global_batch": 1, "seq_len": T},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                            "kind": "oracle",
                            "sample": "each step: the full %d-token layer prefill on the "
                                      "fp64 oracle" % T},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--T", type=int, default=4096)
    ap.add_argument("--decode-n", type=int, default=256)
    ap.add_argument("--cpu-samples", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--legs", default="prefill,decode,e2e,multiseq",
                    help="comma list of legs to run (profiling runs pick one); "
                         "'multiseq' times the chunk scan on packed multi-sequence batches")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
