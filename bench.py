#!/usr/bin/env python
"""Benchmark of the W12 verify path on one GB300 (or N replicas under torchrun).

A step is one verify pass of the 27B-class dense block at M = 16 draft-tree
rows: the four W12 decode-fused GEMMs (fused QKV 7168x5120, O 5120x5120,
gate/up 34816x5120, down 5120x17408) launched in dependency order.  Weights
are generated on the device from the seeded generator, W12-encoded once
(offline, untimed) and stay resident; the block's 506 MB of W12 records is
larger than L2, so no flush is needed between steps.

The JSON line reports decoded-weight GB/s (2 bytes per weight per step), the
roofline of the GEMM kernel against the measured HBM copy bandwidth, the
end-to-end figure through the public API with host buffers, the CPU oracle
timed on a bounded sample, SM clocks sampled during the timed region, and
(under "rows") the other hot-path rows timed in the same run: the Q8 pass over
the same block, the 151936x5120 LM head with fused argmax and tree acceptance,
the 64-layer stack at M=32 (exact and Q8 passes, Q-vs-exact agreement), the
two-level verification step (Q pass, splice, exact pass on 32-node trees), the
block and head at M=192 with 24 trees, and a node budget shared by 24 requests
against per-request trees of the same size (accepted tokens).

--impl reference times the CPU oracle (the plain C reference of the method)
on the same workload and metric, a bounded sample of rows per step.
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

BLOCK = [("qkv", 7168, 5120), ("o", 5120, 5120), ("gate_up", 34816, 5120), ("down", 5120, 17408)]
LMHEAD = (151936, 5120)
WORKLOAD = ("27B-class dense block: fused QKV 7168x5120, O 5120x5120, gate/up 34816x5120, "
            "down 5120x17408; W12 weights (per-channel N(0,s_c), s_c log-uniform [0.005,0.05], "
            "0.5% outliers x2^9, 0.2% zeros, 0.1% denormals); M=16 bf16 N(0,1) rows")
HBM_FALLBACK = 6800.0
# the same metric on both arms (the driver divides one by the other)
METRIC = "W12 verify-GEMM decoded-weight GB/s (27B-class block, M=16)"
# dram__bytes_read.sum + dram__bytes_write.sum of one gate/up launch (34816x5120, M=16)
# from an ncu capture, with the SHA-256 of the GEMM kernel's sources it was taken on: the
# line reports the traffic only while those sources are unchanged.
TRAFFIC_GATE_UP_M16 = 273648896 + 4253696
TRAFFIC_SOURCES_SHA256 = "cdf8af2e23f63f0522e401ba7f4510d5b381c677d4875ca97d002cd59879b4a1"
GEMM_SOURCES = ("lossless_bit_weights_gb300/csrc/w12_gemm.cu", "lossless_bit_weights_gb300/csrc/w12_internal.cuh")


def gemm_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    return h.hexdigest()


def roofline_traffic():
    """The captured traffic of the gate/up launch if the GEMM sources are the captured ones."""
    return TRAFFIC_GATE_UP_M16 if gemm_sources_sha256() == TRAFFIC_SOURCES_SHA256 else None


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["w12", "reference"], default="w12")
    p.add_argument("--M", type=int, default=16)
    p.add_argument("--no-rows", action="store_true", help="skip the extra hot-path rows")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-stack", action="store_true", help="skip the 64-layer stack rows (32 GB of W12)")
    p.add_argument("--only", choices=[n for n, _, _ in BLOCK] + ["lmhead", "cert", "gdn", "wy"], default=None,
                   help="profiling case: repeat one matrix's GEMM (or the LM head) and print its time")
    p.add_argument("--q8", action="store_true", help="with --only: the 8-bit-view GEMM")
    return p.parse_args()


def run_only(args):
    """One matrix, repeated: the small case ncu captures (one kernel, few launches)."""
    import numpy as np
    import torch

    import lossless_bit_weights_gb300 as w12
    import synth

    torch.cuda.set_device(0)
    M = args.M
    if args.only in ("gdn", "wy"):
        # path verify of a 32-node tree and the commit of four accepted nodes on one
        # gated-delta-rule layer of 32 heads of 128 x 128 state
        nn, Hg, dg = 32, 32, 128
        rg = np.random.default_rng(48)
        par = torch.from_numpy(np.array([-1] + [int(rg.integers(max(0, i - 4), i)) for i in range(1, nn)],
                                        np.int32)).cuda()

        def bf16_dev(a):
            u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
            return torch.from_numpy(((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16).view(np.int16)).cuda()

        kk = rg.standard_normal((nn, Hg, dg))
        S = torch.from_numpy((rg.standard_normal((Hg, dg, dg)) * 0.5).astype(np.float32)).cuda()
        q = bf16_dev(rg.standard_normal((nn, Hg, dg)) / np.sqrt(dg))
        k = bf16_dev(kk / np.linalg.norm(kk, axis=2, keepdims=True))
        v = bf16_dev(rg.standard_normal((nn, Hg, dg)))
        al = torch.from_numpy(rg.uniform(0.85, 1.0, (nn, Hg)).astype(np.float32)).cuda()
        be = torch.from_numpy(rg.uniform(0.1, 0.9, (nn, Hg)).astype(np.float32)).cuda()
        O = torch.empty((nn, Hg, dg), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        pn = torch.zeros(nn, dtype=torch.int32, device="cuda")
        node = 0
        for t in range(1, 5):
            kids = [i for i in range(nn) if int(par[i]) == node]
            if not kids:
                break
            node = kids[0]
            pn[t] = node
        pl = torch.tensor([int((pn > 0).sum())], dtype=torch.int32, device="cuda")

        def step():
            if args.only == "wy":
                w12.gdn_wy_verify(S, q, k, v, al, be, par, O=O, status=st)
                return
            w12.gdn_path_verify(S, q, k, v, al, be, par, O=O, status=st)
            w12.gdn_commit(S, k, v, al, be, pl, pn, status=st)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            step()
        b.record()
        torch.cuda.synchronize()
        print(json.dumps({"only": args.only, "us_per_layer": 1e3 * a.elapsed_time(b) / args.steps,
                          "status": int(st.item())}), flush=True)
        return
    if args.only == "cert":
        # certified INT8 head on the head recipe, M rows pointing at random tokens
        V, K = LMHEAD
        W = torch.empty((V, K), dtype=torch.int16, device="cuda")
        synth.weights_dev(0, 0, 9, W, outliers=False)
        H, A = w12.i8_encode(W), w12.encode(W)
        del W
        torch.cuda.empty_cache()
        tgt = np.random.default_rng(16).integers(0, V, M)
        x = torch.from_numpy(synth.peaked_activations(1, 0, 101, synth.weight_rows(0, 0, 9, K, tgt, outliers=False),
                                                      8.0).view(np.int16)).cuda()
        ws = w12.Workspace()
        for _ in range(args.warmup):
            tok, nc = w12.w12_cert_head_argmax(x, H, A, ws=ws)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            tok, nc = w12.w12_cert_head_argmax(x, H, A, ws=ws)
        b.record()
        torch.cuda.synchronize()
        print(json.dumps({"only": "cert", "M": M, "V": V, "K": K, "us": 1e3 * a.elapsed_time(b) / args.steps,
                          "ncand": nc.cpu().tolist()}), flush=True)
        return
    if args.only == "lmhead":
        tensor, (N, K) = 9, LMHEAD
    else:
        tensor = [n for n, _, _ in BLOCK].index(args.only)
        _, N, K = BLOCK[tensor]
    W = torch.empty((N, K), dtype=torch.int16, device="cuda")
    synth.weights_dev(0, 0, tensor, W)
    A = w12.encode(W)
    del W
    torch.cuda.empty_cache()
    x = torch.empty((M, K), dtype=torch.int16, device="cuda")
    synth.activations_dev(1, 0, tensor, x)
    ws = w12.Workspace()
    if args.only == "lmhead":
        fn = lambda: w12.w12_lmhead_argmax(x, A, q8=args.q8, ws=ws)
    else:
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        fn = lambda: (w12.w12_gemm_q8 if args.q8 else w12.w12_gemm)(x, A, y=y, ws=ws)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    us = 1e3 * a.elapsed_time(b) / args.steps
    sb = A.stream_bytes(q8=args.q8) + 2 * M * K + 4 * M * N
    print(json.dumps({"only": args.only, "q8": args.q8, "M": M, "N": N, "K": K, "us": us,
                      "stream_GBps": sb / us / 1e3, "decoded_GBps": 2 * N * K / us / 1e3}), flush=True)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK, "fallback"


# ------------------------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), hw=parts[5], hwt=parts[6], swt=parts[7],
                                 pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                          ("pcap", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in rows):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------ distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------ CPU oracle timing

def oracle_block_sample(M: int, rows_per_matrix: int, layer: int = 0, threads: int | None = None):
    """Oracle work on a bounded sample of the block: decode (from the canonical
    W12 planes) and fp64 GEMM of `rows_per_matrix` channels of each matrix.
    Returns (seconds, weights processed, threads used)."""
    import numpy as np

    import oracle
    import synth

    threads = threads or (os.cpu_count() or 1)
    prepared = []
    for tensor, (_, N, K) in enumerate(BLOCK):
        rows = np.arange(rows_per_matrix) * (N // rows_per_matrix)
        W = synth.weight_rows(0, layer, tensor, K, rows)
        prepared.append((oracle.encode(W), synth.activations(1, layer, tensor, M, K)))
    t0 = time.perf_counter()
    n = 0
    for enc, x in prepared:
        Wd = oracle.decode(enc)
        oracle.gemm(x, Wd, threads=threads, with_bound=False)
        n += Wd.size
    return time.perf_counter() - t0, n, threads


def calibrate_rows(M: int, target_s: float) -> int:
    rows = 64
    dt, _, _ = oracle_block_sample(M, rows)
    while dt < target_s / 4 and rows < 8192:
        rows *= 2
        dt, _, _ = oracle_block_sample(M, rows)
    return max(32, int(rows * target_s / max(dt, 1e-3)))


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: each step decodes and multiplies a
    bounded sample of the block's channels at M rows."""
    if rank != 0:
        return
    rows = calibrate_rows(args.M, target_s=0.25)
    for _ in range(args.warmup):
        oracle_block_sample(args.M, rows)
    total_t, total_w = 0.0, 0
    threads = os.cpu_count() or 1
    for _ in range(args.steps):
        dt, n, threads = oracle_block_sample(args.M, rows)
        total_t += dt
        total_w += n
    value = 2.0 * total_w / total_t / 1e9
    sample = f"{rows} channels of each block matrix per step (decode + fp64 GEMM at M={args.M})"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": args.M, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------ GPU arm

def encode_block(w12, synth, torch, layer: int):
    mats = []
    for tensor, (name, N, K) in enumerate(BLOCK):
        W = torch.empty((N, K), dtype=torch.int16, device="cuda")
        synth.weights_dev(0, layer, tensor, W)
        A = w12.encode(W)
        del W
        mats.append((name, A))
    torch.cuda.empty_cache()
    return mats


def run_w12(args, world, rank, local):
    import torch

    import lossless_bit_weights_gb300 as w12
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    M = args.M
    mats = encode_block(w12, synth, torch, layer=0)
    xs, ys = [], []
    for tensor, (name, A) in enumerate(mats):
        x = torch.empty((M, A.K), dtype=torch.int16, device=dev)
        synth.activations_dev(1, 0, tensor, x)
        xs.append(x)
        ys.append(torch.empty((M, A.N), dtype=torch.float32, device=dev))
    ws = w12.Workspace(dev)
    ws.get(max(w12.gemm_workspace_size(M, A.N, A.K) for _, A in mats))
    weights = sum(A.N * A.K for _, A in mats)
    stream_bytes = sum(A.stream_bytes() + 2 * M * A.K + 4 * M * A.N for _, A in mats)
    stored = sum(A.stored_bytes() for _, A in mats)
    n_esc = sum(A.n_esc for _, A in mats)

    def step():
        for (_, A), x, y in zip(mats, xs, ys):
            w12.w12_gemm(x, A, y=y, ws=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- timed region: K steps back to back, events only at the two ends, so a GEMM
    # streams its weights while the previous one drains (programmatic dependent launch)
    K = args.steps
    s = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(s)
    for k in range(K):
        step()
    t1.record(s)
    torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world)

    # ---- second timed pass: an event before and after every launch, for the per-matrix
    # times and the roofline of the largest launch (gate/up).  The events stop one launch
    # overlapping the next, so these per-launch times are upper bounds.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(mats) + 1)] for _ in range(K)]
    torch.cuda.synchronize()
    for k in range(K):
        e = evs[k]
        for i, ((_, A), x, y) in enumerate(zip(mats, xs, ys)):
            e[i].record(s)
            w12.w12_gemm(x, A, y=y, ws=ws)
        e[len(mats)].record(s)
    torch.cuda.synchronize()
    per_mat_ms = [statistics.fmean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(K)) for i in range(len(mats))]

    # ---- the dominant launch alone, back to back (as in a stream of such launches): its
    # average duration for the roofline
    gi = [n for n, _ in mats].index("gate_up")
    Ag, xg, yg = mats[gi][1], xs[gi], ys[gi]
    ng = max(20, K // 4)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    g0.record(s)
    for _ in range(ng):
        w12.w12_gemm(xg, Ag, y=yg, ws=ws)
    g1.record(s)
    torch.cuda.synchronize()
    clk = clocks.stop()
    gate_ms = g0.elapsed_time(g1) / ng

    value = world * 2.0 * weights * K / (elapsed_ms * 1e-3) / 1e9
    hbm, hbm_kind = peaks()
    gate_bytes = Ag.stream_bytes() + 2 * M * Ag.K + 4 * M * Ag.N
    achieved = gate_bytes / (gate_ms * 1e-3) / 1e9
    achieved_block = stream_bytes / (elapsed_ms / K * 1e-3) / 1e9

    # ---- end to end through the public API with pinned host buffers.  Every step copies its
    # inputs in and its outputs out; a copy stream does that one step ahead (inputs) and one
    # behind (outputs) while the compute stream runs the step's GEMMs back to back, with
    # double-buffered device inputs and outputs.  The timed region holds every copy,
    # including the last step's outputs.
    xh = [torch.empty_like(x, device="cpu").pin_memory() for x in xs]
    for x, h in zip(xs, xh):
        h.copy_(x.cpu())
    yh = [torch.empty_like(y, device="cpu").pin_memory() for y in ys]
    xb = [[x, torch.empty_like(x)] for x in xs]
    yb = [[y, torch.empty_like(y)] for y in ys]
    cs = torch.cuda.Stream()
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]     # inputs of buffer b loaded, outputs of b read
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]   # GEMMs on buffer b finished

    def e2e_run(n_steps):
        with torch.cuda.stream(cs):
            for x, h in zip(xb, xh):
                x[0].copy_(h, non_blocking=True)
            ev_in[0].record(cs)
        for step in range(n_steps):
            b = step & 1
            s.wait_event(ev_in[b])
            for (_, A), x, y in zip(mats, xb, yb):
                w12.w12_gemm(x[b], A, y=y[b], ws=ws)
            ev_done[b].record(s)
            with torch.cuda.stream(cs):
                if step >= 1:                       # the previous step's outputs
                    cs.wait_event(ev_done[b ^ 1])
                    for y, hy in zip(yb, yh):
                        hy.copy_(y[b ^ 1], non_blocking=True)
                if step + 1 < n_steps:              # the next step's inputs (after the GEMMs of step - 1)
                    for x, h in zip(xb, xh):
                        x[b ^ 1].copy_(h, non_blocking=True)
                ev_in[b ^ 1].record(cs)
        with torch.cuda.stream(cs):                 # the last step's outputs
            cs.wait_event(ev_done[(n_steps - 1) & 1])
            for y, hy in zip(yb, yh):
                hy.copy_(y[(n_steps - 1) & 1], non_blocking=True)
            ev_in[0].record(cs)
        s.wait_event(ev_in[0])

    e2e_run(3)
    torch.cuda.synchronize()
    # the pipelined outputs are the plain path's
    for (_, A), x, y, hy in zip(mats, xs, ys, yh):
        w12.w12_gemm(x, A, y=y, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(hy, y.cpu()), "pipelined end-to-end outputs differ"
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    Ke = max(1, K // 2)
    e2e_run(Ke)
    e1.record(s)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    h2d = sum(x.numel() * 2 for x in xs)
    d2h = sum(y.numel() * 4 for y in ys)
    e2e = {"value": world * 2.0 * weights * Ke / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "copies": "a copy stream, one step ahead (inputs) and behind (outputs)"}

    rows = None
    if not args.no_rows:
        rows = extra_rows(w12, synth, torch, mats, xs, ws, M, args, hbm)

    del mats
    torch.cuda.empty_cache()
    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        r = calibrate_rows(M, target_s=2.0)
        dt, n, threads = oracle_block_sample(M, r)
        cpu = {"value": 2.0 * n / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{r} channels of each block matrix: decode + fp64 GEMM at M={M} ({dt:.1f} s wall)"}

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "weights_per_step": weights, "stored_bytes": stored,
                       "bits_per_weight": 8.0 * stored / weights, "escape_fraction": n_esc / weights,
                       "us_per_layer": 1e3 * elapsed_ms / K, "parallelism": f"replicas x{world}",
                       "l2": "no flush: 506 MB of W12 per step, larger than the 129 MB L2"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": roofline_traffic(), "peak_kind": hbm_kind,
                         "kernel": "k_gemm_tc<NT=16,Q8=0,mode=pair,EPI=store>, gate/up launch (34816x5120, M=16)",
                         "algorithmic_bytes": gate_bytes, "launch_us": 1e3 * gate_ms,
                         "timing": "gate/up alone, back to back, CUDA events around the loop",
                         "block_achieved": achieved_block, "block_frac": achieved_block / hbm,
                         "per_matrix_us_event_bracketed": {n: 1e3 * t for (n, _), t in zip(BLOCK_NAMES, per_mat_ms)}},
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")} | {"samples": clk["samples"]},
            "gpu_launches": len(BLOCK) * K,  # launches of the timed region (the step loop)
        }
        if rows is not None:
            line["rows"] = rows
        print(json.dumps(line), flush=True)


BLOCK_NAMES = [(n, (N, K)) for n, N, K in BLOCK]


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(path))["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def timed_ms(torch, fn, n, warm=3):
    """Average ms of fn over n back-to-back calls, CUDA events around the loop."""
    s = torch.cuda.current_stream()
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(n):
        fn()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def graph_ms(torch, fn, n, warm=3):
    """Average ms of one replay of a CUDA graph that holds one call of fn (device time of
    a launch sequence whose kernels are shorter than the host's launch overhead)."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(n):
        g.replay()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def gemm_bytes(A, M, q8=False):
    return A.stream_bytes(q8=q8) + 2 * M * A.K + 4 * M * A.N


def extra_rows(w12, synth, torch, mats, xs, ws, M, args, hbm):
    """The other hot-path rows, each timed with CUDA events (not part of `value`):
    the Q8 pass over the block at M=16, the LM head with fused argmax + acceptance at
    M=16, the 64-layer stack at M=32 (exact and Q8 passes, then the W12 head with a
    32-node tree), and the block and head at M=192 with 24 eight-node trees."""
    import numpy as np
    out = {}
    steps = max(5, args.steps // 4)
    dev = torch.device("cuda", torch.cuda.current_device())

    # ---- Q8 pass over the block at M = 16
    ysq = [torch.empty((M, A.N), dtype=torch.float32, device=dev) for _, A in mats]

    def q8_step():
        for (_, A), x, y in zip(mats, xs, ysq):
            w12.w12_gemm_q8(x, A, y=y, ws=ws)

    ms = timed_ms(torch, q8_step, steps)
    weights = sum(A.N * A.K for _, A in mats)
    qbytes = sum(gemm_bytes(A, M, True) for _, A in mats)
    out["q8_block_m16"] = {"us": 1e3 * ms, "decoded_GBps": 2 * weights / (ms * 1e-3) / 1e9,
                           "stream_GBps": qbytes / (ms * 1e-3) / 1e9, "frac_hbm": qbytes / (ms * 1e-3) / 1e9 / hbm}

    # ---- the LM head (151936 x 5120), W12-encoded once
    V, K = LMHEAD
    W = torch.empty((V, K), dtype=torch.int16, device=dev)
    synth.weights_dev(0, 0, 9, W)
    H = w12.encode(W)
    del W
    torch.cuda.empty_cache()
    ws2 = w12.Workspace(dev)

    def head_case(Mh, xseed_tensor, n_req, nodes):
        x = torch.empty((Mh, K), dtype=torch.int16, device=dev)
        synth.activations_dev(1, 0, xseed_tensor, x)
        parent = np.concatenate([synth.tree(2, r, nodes, nodes) for r in range(n_req)]).astype(np.int32)
        draft = np.concatenate([synth.drafts(3, r, nodes, nodes, V) for r in range(n_req)]).astype(np.int32)
        offsets = None if n_req == 1 else torch.from_numpy(np.arange(0, Mh + 1, nodes, dtype=np.int32)).to(dev)
        p, d = torch.from_numpy(parent).to(dev), torch.from_numpy(draft).to(dev)
        fn = lambda: w12.w12_lmhead_verify(x, H, p, d, req_offsets=offsets, ws=ws2)
        return x, fn

    x16, fn = head_case(M, 9, 1, M)
    ms = timed_ms(torch, fn, steps)
    hb = H.stream_bytes() + 2 * M * K
    out["lmhead_verify_m16"] = {"us": 1e3 * ms, "decoded_GBps": 2 * V * K / (ms * 1e-3) / 1e9,
                                "stream_GBps": hb / (ms * 1e-3) / 1e9, "frac_hbm": hb / (ms * 1e-3) / 1e9 / hbm}

    # ---- the 64-layer stack at M = 32: exact pass, Q8 pass, then the head + 32-node tree
    if not args.no_stack:
        Ms, layers = 32, 64
        stack = [encode_block(w12, synth, torch, layer) for layer in range(layers)]
        xs32, ys32 = [], []
        for tensor, (_, A) in enumerate(stack[0]):
            x = torch.empty((Ms, A.K), dtype=torch.int16, device=dev)
            synth.activations_dev(1, 0, tensor, x)
            xs32.append(x)
            ys32.append(torch.empty((Ms, A.N), dtype=torch.float32, device=dev))
        ws3 = w12.Workspace(dev)
        ws3.get(max(w12.gemm_workspace_size(Ms, A.N, A.K) for _, A in stack[0]))

        def pass_(q8):
            f = w12.w12_gemm_q8 if q8 else w12.w12_gemm
            for blk in stack:
                for (_, A), x, y in zip(blk, xs32, ys32):
                    f(x, A, y=y, ws=ws3)

        n_pass = max(3, steps // 10)
        w_stack = sum(A.N * A.K for blk in stack for _, A in blk)
        stored = sum(A.stored_bytes() for blk in stack for _, A in blk)
        n_esc = sum(A.n_esc for blk in stack for _, A in blk)
        row = {}
        for q8 in (False, True):
            ms = timed_ms(torch, lambda: pass_(q8), n_pass, warm=1)
            sb = sum(gemm_bytes(A, Ms, q8) for blk in stack for _, A in blk)
            row["q8" if q8 else "exact"] = {
                "ms_per_pass": ms, "us_per_layer": 1e3 * ms / layers,
                "decoded_GBps": 2 * w_stack / (ms * 1e-3) / 1e9, "stream_GBps": sb / (ms * 1e-3) / 1e9,
                "frac_hbm": sb / (ms * 1e-3) / 1e9 / hbm}
        out["stack64_m32"] = {"layers": layers, "weights": w_stack, "stored_bytes": stored,
                              "bits_per_weight": 8.0 * stored / w_stack, "escape_fraction": n_esc / w_stack,
                              **row}
        # config 3: Q8 stack pass, then the W12 head with argmax + 32-node tree acceptance
        x32, fn32 = head_case(Ms, 9, 1, Ms)
        ms_head = timed_ms(torch, fn32, steps)
        ms_q = row["q8"]["ms_per_pass"]
        # Q-vs-exact top-1 agreement of the head: the 32 rows plus 1024 more seeded rows
        xa = torch.empty((1024, K), dtype=torch.int16, device=dev)
        synth.activations_dev(1, 0, 11, xa)
        agree, total = 0, 0
        for xx in (x32, xa):
            te = w12.w12_lmhead_argmax(xx, H, ws=ws2)
            tq = w12.w12_lmhead_argmax(xx, H, q8=True, ws=ws2)
            agree += int((te == tq).sum())
            total += xx.shape[0]
        out["q8_stack64_m32_head_tree32"] = {
            "q8_pass_ms": ms_q, "head_verify_us": 1e3 * ms_head, "total_ms": ms_q + ms_head,
            "q_vs_exact_top1_agreement": agree / total, "agreement_rows": total}

        # two-level verification step: Q pass (8-bit view of the stack and the head) on a
        # 32-node tree, splice of its accepted path + bonus + a subtree drafted again into a
        # 32-node tree, exact pass (W12 stack and head) on that tree
        n = Ms
        rng = np.random.default_rng(7)
        tq0 = w12.w12_lmhead_argmax(x32, H, q8=True, ws=ws2).cpu().numpy()
        pq = synth.tree(2, 7, n, n)
        dq = synth.drafts(3, 7, n, n, V)
        for i in range(1, n):
            if rng.random() < 0.7:
                dq[i] = tq0[pq[i]]
        sp = np.array([-1 if j == 0 or rng.random() < 0.3 else int(rng.integers(0, j)) for j in range(n - 2)], np.int32)
        sd = synth.drafts(3, 8, n, n - 2, V)
        pq_d, dq_d = torch.from_numpy(pq).to(dev), torch.from_numpy(dq).to(dev)
        sp_d, sd_d = torch.from_numpy(sp).to(dev), torch.from_numpy(sd).to(dev)
        xs_new = torch.empty((n - 1, K), dtype=torch.int16, device=dev)
        synth.activations_dev(1, 0, 13, xs_new)
        lens = {}

        def tlv_step():
            pass_(True)
            _, pl, pn, bo = w12.w12_lmhead_verify(x32, H, pq_d, dq_d, q8=True, ws=ws2)
            par, dr, _, xe = w12.tlv_splice(pl, pn, bo, dq_d, x32, sp_d, sd_d, xs_new, n)
            pass_(False)
            _, pl2, _, _ = w12.w12_lmhead_verify(xe, H, par, dr, ws=ws2)
            lens["q"], lens["exact"] = pl, pl2

        ms_tlv = timed_ms(torch, tlv_step, n_pass, warm=1)
        # the splice alone, 20 calls captured in a CUDA graph (a call from Python takes longer
        # to issue than the kernel takes to run)
        pn0 = torch.zeros(n, dtype=torch.int32, device=dev)
        bo0 = torch.zeros(1, dtype=torch.int32, device=dev)
        splice = lambda: w12.tlv_splice(lens["q"], pn0, bo0, dq_d, x32, sp_d, sd_d, xs_new, n)
        splice()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(20):
                splice()
        ms_splice = timed_ms(torch, graph.replay, 10) / 20
        out["tlv_step_stack64_m32"] = {"ms_per_step": ms_tlv, "splice_us": 1e3 * ms_splice,
                                       "q_path_len": int(lens["q"][0]), "exact_path_len": int(lens["exact"][0]),
                                       "tree_nodes": n}
        del stack
        torch.cuda.empty_cache()

    # ---- M = 192: the block and the head, 24 requests x 8 nodes
    Mb = 192
    xb, yb = [], []
    for tensor, (_, A) in enumerate(mats):
        x = torch.empty((Mb, A.K), dtype=torch.int16, device=dev)
        synth.activations_dev(1, 1, tensor, x)
        xb.append(x)
        yb.append(torch.empty((Mb, A.N), dtype=torch.float32, device=dev))
    ws4 = w12.Workspace(dev)
    ws4.get(max(w12.gemm_workspace_size(Mb, A.N, A.K) for _, A in mats))

    def blk192():
        for (_, A), x, y in zip(mats, xb, yb):
            w12.w12_gemm(x, A, y=y, ws=ws4)

    ms_b = timed_ms(torch, blk192, steps)
    x192, fn192 = head_case(Mb, 10, 24, 8)
    ms_h = timed_ms(torch, fn192, steps)
    tf, tf_kind = bf16_peak()
    b_bytes = sum(gemm_bytes(A, Mb) for _, A in mats)
    h_bytes = H.stream_bytes() + 2 * Mb * K
    b_flops = sum(2.0 * Mb * A.N * A.K for _, A in mats)
    h_flops = 2.0 * Mb * V * K

    def roof(ms, nbytes, flops):
        t_hbm = nbytes / (hbm * 1e9) * 1e3
        t_tc = flops / (tf * 1e12) * 1e3
        return {"us": 1e3 * ms, "hbm_floor_us": 1e3 * t_hbm, "tensor_floor_us": 1e3 * t_tc,
                "frac_of_binding_roofline": max(t_hbm, t_tc) / ms,
                "binding": "hbm" if t_hbm >= t_tc else "tensor",
                "tflops": flops / (ms * 1e-3) / 1e12, "stream_GBps": nbytes / (ms * 1e-3) / 1e9}

    out["block_head_m192_24trees"] = {"block": roof(ms_b, b_bytes, b_flops), "head_verify": roof(ms_h, h_bytes, h_flops),
                                      "total_us": 1e3 * (ms_b + ms_h), "tensor_peak_tflops": tf,
                                      "tensor_peak_kind": tf_kind}

    # ---- node budget shared across 24 requests vs per-request trees of the same total size.
    # Synthetic drafter: 32 candidate nodes per request; the children of a node carry
    # distinct draft tokens whose confidences (each request its own level, halving from the
    # first child on, summing below 1) are the probabilities that each one is the target's
    # token; at most one child matches.  The root is the committed token (confidence 1), so
    # a node's path score is the probability that it is accepted and the shared top-192
    # maximises the expected accepted length.  The kept nodes go through the head and
    # acceptance; accepted tokens averaged over seeds.
    n_req, cand, B = 24, 32, 192
    C = n_req * cand
    xc = torch.empty((C, K), dtype=torch.int16, device=dev)
    synth.activations_dev(1, 2, 14, xc)
    t_all = torch.cat([w12.w12_lmhead_argmax(xc[i:i + 256], H, ws=ws2) for i in range(0, C, 256)]).cpu().numpy()
    off_c = torch.from_numpy(np.arange(0, C + 1, cand, dtype=np.int32)).to(dev)
    acc = {"shared": [], "per_request": []}
    for trial in range(8):
        rng = np.random.default_rng(1000 + trial)
        par_c = np.concatenate([synth.tree(2, 500 + 24 * trial + r, cand, cand) for r in range(n_req)]).astype(np.int32)
        level = rng.uniform(0.4, 0.95, n_req)
        conf_c = np.ones(C, np.float32)
        dr_c = rng.integers(0, V, C).astype(np.int32)
        for r in range(n_req):
            r0 = r * cand
            kids = [[] for _ in range(cand)]
            for i in range(1, cand):
                kids[par_c[r0 + i]].append(i)
            for pn, ch in enumerate(kids):
                tp = t_all[r0 + pn]
                u, cum = rng.random(), 0.0
                for k, i in enumerate(ch):
                    conf_c[r0 + i] = np.float32(level[r] * 0.5 ** (k + 1) * rng.uniform(0.8, 1.0))
                    lo = cum
                    cum += float(conf_c[r0 + i])
                    if lo <= u < cum:
                        dr_c[r0 + i] = tp                           # this child is the target's token
                    elif dr_c[r0 + i] == tp:
                        dr_c[r0 + i] = (tp + 1 + k) % V             # the others are not
        p_d, c_d, d_d = (torch.from_numpy(a).to(dev) for a in (par_c, conf_c, dr_c))
        for name, budget, per in (("shared", B, False), ("per_request", B // n_req, True)):
            po, do, so, oo, nk = w12.tree_budget_select(p_d, c_d, d_d, off_c, budget, per)
            xs = w12.gather_rows(xc, so, B)
            _, pl, _, _ = w12.w12_lmhead_verify(xs, H, po[:B], do[:B], req_offsets=oo, ws=ws2)
            acc[name].append(int(pl.sum()))

        def budget_step():
            po, do, so, oo, nk = w12.tree_budget_select(p_d, c_d, d_d, off_c, B, False)
            xs = w12.gather_rows(xc, so, B)
            w12.w12_lmhead_verify(xs, H, po[:B], do[:B], req_offsets=oo, ws=ws2)

    ms_bud = timed_ms(torch, budget_step, steps)
    sh, pr = float(np.mean(acc["shared"])), float(np.mean(acc["per_request"]))
    out["shared_budget_24x8"] = {"accepted_tokens_shared": sh, "accepted_tokens_per_request": pr,
                                 "gain": sh / pr - 1.0 if pr else None, "trials": len(acc["shared"]),
                                 "candidates": C, "budget": B, "select_gather_verify_us": 1e3 * ms_bud}
    del H
    torch.cuda.empty_cache()

    # ---- certified INT8 head against the W12 head on the same weights: the head recipe
    # (no x2^9 outliers, which would set every channel's INT8 scale) and 16 rows pointing
    # at random tokens (a verify pass's final hidden state points at the token it
    # predicts); then 16 plain N(0,1) rows, where no logit stands out.
    W = torch.empty((V, K), dtype=torch.int16, device=dev)
    synth.weights_dev(0, 0, 9, W, outliers=False)
    Hc, Ac = w12.i8_encode(W), w12.encode(W)
    del W
    torch.cuda.empty_cache()
    tgt = np.random.default_rng(16).integers(0, V, M)
    rows = synth.weight_rows(0, 0, 9, K, tgt, outliers=False)
    cert = {"rows": M, "beta": 8.0, "weights": "head recipe (no x2^9 outliers)"}
    xn = torch.empty((M, K), dtype=torch.int16, device=dev)
    synth.activations_dev(1, 0, 103, xn)
    xp = torch.from_numpy(synth.peaked_activations(1, 0, 101, rows, 8.0).view(np.int16)).to(dev)
    for name, xr in (("peaked", xp), ("isotropic", xn)):
        tok_c, nc = w12.w12_cert_head_argmax(xr, Hc, Ac, ws=ws2)
        tok_w = w12.w12_lmhead_argmax(xr, Ac, ws=ws2)
        ms_w = timed_ms(torch, lambda: w12.w12_lmhead_argmax(xr, Ac, ws=ws2), steps)
        ms_c = timed_ms(torch, lambda: w12.w12_cert_head_argmax(xr, Hc, Ac, ws=ws2), steps)
        nc = nc.cpu().numpy()
        cert[name] = {"w12_head_us": 1e3 * ms_w, "cert_int8_head_us": 1e3 * ms_c, "speedup": ms_w / ms_c,
                      "candidates_mean": float(nc.mean()), "candidates_max": int(nc.max()),
                      "same_tokens_as_w12_head": bool(torch.equal(tok_c, tok_w)),
                      "int8_stream_GBps": (Hc.stream_bytes() + 2 * M * K) / (ms_c * 1e-3) / 1e9,
                      "w12_stream_GBps": (Ac.stream_bytes() + 2 * M * K) / (ms_w * 1e-3) / 1e9}
        if name == "peaked":
            cert[name]["rows_on_target"] = int((tok_c.cpu().numpy() == tgt).sum())
    out["cert_head_m16"] = cert
    del Hc, Ac
    torch.cuda.empty_cache()

    # ---- recurrent layers of a hybrid target: 48 gated-delta-rule layers, 32 heads of
    # 128 x 128 float state, a 32-node draft tree.  One step: path verify of every node on
    # every layer, then the commit of the accepted path (the same four nodes) into every
    # layer's state.  Per-node state snapshots would hold n x H x dv x dk floats per layer.
    n_l, Hg, dg, nn = 48, 32, 128, 32
    rg = np.random.default_rng(48)
    par_g = torch.from_numpy(np.array([-1] + [int(rg.integers(max(0, i - 4), i)) for i in range(1, nn)],
                                      np.int32)).to(dev)

    def bf16_dev(a):
        u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
        return torch.from_numpy(((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16).view(np.int16)).to(dev)

    layers_g = []
    for _ in range(n_l):
        kk = rg.standard_normal((nn, Hg, dg))
        layers_g.append(dict(
            S=torch.from_numpy((rg.standard_normal((Hg, dg, dg)) * 0.5).astype(np.float32)).to(dev),
            q=bf16_dev(rg.standard_normal((nn, Hg, dg)) / np.sqrt(dg)),
            k=bf16_dev(kk / np.linalg.norm(kk, axis=2, keepdims=True)),
            v=bf16_dev(rg.standard_normal((nn, Hg, dg))),
            a=torch.from_numpy(rg.uniform(0.85, 1.0, (nn, Hg)).astype(np.float32)).to(dev),
            b=torch.from_numpy(rg.uniform(0.1, 0.9, (nn, Hg)).astype(np.float32)).to(dev),
            O=torch.empty((nn, Hg, dg), dtype=torch.float32, device=dev)))
    acc_nodes = [0]
    while len(acc_nodes) < 5:                      # a path of four accepted draft nodes
        kids = [i for i in range(nn) if int(par_g[i]) == acc_nodes[-1]]
        if not kids:
            break
        acc_nodes.append(kids[0])
    pn = torch.zeros(nn, dtype=torch.int32, device=dev)
    pn[:len(acc_nodes)] = torch.tensor(acc_nodes, dtype=torch.int32)
    pl = torch.tensor([len(acc_nodes) - 1], dtype=torch.int32, device=dev)
    st_g = torch.zeros(1, dtype=torch.int32, device=dev)
    S_keep = [Lg["S"].clone() for Lg in layers_g]

    def gdn_verify_all():
        for Lg in layers_g:
            w12.gdn_path_verify(Lg["S"], Lg["q"], Lg["k"], Lg["v"], Lg["a"], Lg["b"], par_g, O=Lg["O"], status=st_g)

    def gdn_commit_all():
        for Lg in layers_g:
            w12.gdn_commit(Lg["S"], Lg["k"], Lg["v"], Lg["a"], Lg["b"], pl, pn, status=st_g)

    def gdn_wy_all():
        for Lg in layers_g:
            w12.gdn_wy_verify(Lg["S"], Lg["q"], Lg["k"], Lg["v"], Lg["a"], Lg["b"], par_g, O=Lg["O"], status=st_g)

    # 48 launches of a few microseconds each: eager timing measures the host's launch rate,
    # so the device time comes from replaying the 48 launches captured in a CUDA graph
    ms_v_e = timed_ms(torch, gdn_verify_all, steps)
    ms_wy_e = timed_ms(torch, gdn_wy_all, steps)
    ms_v = graph_ms(torch, gdn_verify_all, steps)
    ms_wy = graph_ms(torch, gdn_wy_all, steps)
    ms_c = graph_ms(torch, gdn_commit_all, steps)      # each call advances the states further
    for Lg, S0g in zip(layers_g, S_keep):
        Lg["S"].copy_(S0g)
    # the WY launch's algorithmic bytes: the float state, the node vectors and scalars, the tree
    # and the outputs (the state products are 2 H dv dk 2n flops, small beside the bytes)
    wy_bytes = n_l * (Hg * dg * dg * 4 + nn * Hg * (2 * dg * 2 + dg * 2 + 8) + nn * 4 + nn * Hg * dg * 4)
    out["gdn_verify_48x32"] = {"layers": n_l, "heads": Hg, "dk": dg, "dv": dg, "tree_nodes": nn,
                               "accepted": len(acc_nodes) - 1, "path_verify_us": 1e3 * ms_v,
                               "wy_verify_us": 1e3 * ms_wy, "commit_us": 1e3 * ms_c,
                               "timing": "CUDA-graph replay of the 48 launches",
                               "path_verify_eager_us": 1e3 * ms_v_e, "wy_verify_eager_us": 1e3 * ms_wy_e,
                               "wy_stream_GBps": wy_bytes / (ms_wy * 1e-3) / 1e9,
                               "wy_frac_hbm": wy_bytes / (ms_wy * 1e-3) / 1e9 / hbm,
                               "wy_kernel": "tcgen05 bf16 MMAs over the state's three exact bf16 pieces",
                               "step_us": 1e3 * (min(ms_v, ms_wy) + ms_c),
                               "snapshot_bytes_avoided": n_l * nn * Hg * dg * dg * 4,
                               "status": int(st_g.item())}

    # ---- context: torch bf16 matmul (cuBLAS) over the block's four shapes, the same weights
    # as plain bf16 (2 B per weight, nothing to decode), bf16 outputs, launched back to back
    # like the W12 block on the same inputs; the block's 660 MB of bf16 exceed the L2
    Wb = []
    for tensor, (_, A) in enumerate(mats):
        W = torch.empty((A.N, A.K), dtype=torch.int16, device=dev)
        synth.weights_dev(0, 0, tensor, W)
        Wb.append(W.view(torch.bfloat16))
    wsc = w12.Workspace(dev)
    wsc.get(max(w12.gemm_workspace_size(192, A.N, A.K) for _, A in mats))
    ctx = {"weights": "the block's bf16 weights (layer 0)", "outputs": "bf16 (cuBLAS), fp32 (W12)"}
    for Mc in (16, 32, 192):
        xc = []
        for tensor, (_, A) in enumerate(mats):
            x = torch.empty((Mc, A.K), dtype=torch.int16, device=dev)
            synth.activations_dev(1, 0, tensor, x)
            xc.append(x)
        yb16 = [torch.empty((Mc, A.N), dtype=torch.bfloat16, device=dev) for _, A in mats]
        y32 = [torch.empty((Mc, A.N), dtype=torch.float32, device=dev) for _, A in mats]

        def cublas_block():
            for W, x, y in zip(Wb, xc, yb16):
                torch.mm(x.view(torch.bfloat16), W.t(), out=y)

        def w12_block():
            for (_, A), x, y in zip(mats, xc, y32):
                w12.w12_gemm(x, A, y=y, ws=wsc)

        ms_cb = timed_ms(torch, cublas_block, steps)
        ms_w = timed_ms(torch, w12_block, steps)
        cb_bytes = sum(2 * A.N * A.K + 2 * Mc * A.K + 2 * Mc * A.N for _, A in mats)
        ctx[f"m{Mc}"] = {"cublas_bf16_us": 1e3 * ms_cb, "w12_us": 1e3 * ms_w, "w12_speedup": ms_cb / ms_w,
                         "cublas_stream_GBps": cb_bytes / (ms_cb * 1e-3) / 1e9,
                         "cublas_frac_hbm": cb_bytes / (ms_cb * 1e-3) / 1e9 / hbm}
    out["cublas_bf16_block_context"] = ctx
    del Wb
    torch.cuda.empty_cache()
    return out


def main():
    args = parse_args()
    if args.only:
        run_only(args)
        return
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_w12(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
