#!/usr/bin/env python
"""Benchmark of the batched speculative-decoding verifier on GB300.

One step = one verification call over one batch: the headline workload is the target-only
(one-hot draft) chain with B=64 requests, k=7 drafts, V=128256, bf16 logits (T = 1), i.e.
512 verified positions per step.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): every rank verifies its own batch (weak scaling, no
data-path collective); the host-side barrier and the max of the ranks' times are the only
communication.  --impl reference times the CPU oracle on the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
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

METRIC = "verified positions/sec and HBM GB/s (fraction of GB300 peak) for verify"
UNIT = "positions/s"
WORKLOAD = ("b64k7 target-only chain: B=64 requests, k=7 drafts, V=128256, bf16 logits "
            "~N(0,3^2) with one +8 peak per row, one-hot drafts (target argmax w.p. 0.7), T=1.0")
B, K_DRAFTS, V = 64, 7, 128256
N_SETS = 3  # rotating input sets: 3 x 131 MB > L2 (129 MB)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "verify_call_b64k7_traffic.json")
LAUNCHES_PER_CALL = 2  # sv_stream_kernel, then sv_finalize_kernel (programmatic dependent launch)
GRAPH_CALLS = 30  # verify calls captured in one CUDA graph for the timed region
KV_SETS = 8       # KV-compaction index sets rotated over one pool
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal
KERNEL_SOURCES = [os.path.join(ROOT, "speculative_decoding_verification_verify_gb300", "csrc", f)
                  for f in ("spec_verify.cu", "sv_device.cuh", "sv_draw.cuh", "sv_stream.cuh", "sv_rescan.cuh",
                          "sv_decide.cuh")]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work spent timing the oracle baseline")
    ap.add_argument("--no-modes", action="store_true", help="skip the other verify modes")
    ap.add_argument("--modes", default="all",
                    help="comma list of other modes to time: greedy, tree, block, with_q, b1k3, "
                         "variants, budget, kv_compact (default all)")
    ap.add_argument("--kv-max-pos", type=int, default=512,
                    help="positions per request of the KV-compaction cache (512: 3.2 GB)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    return ap.parse_args()


# --------------------------------------------------------------------------------------------
# Distributed plumbing (host-side only)
# --------------------------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist

            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend, rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float, device) -> float:
        if not self.pg:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def rank_offset(rank: int) -> int:
    """Each rank draws from its own Philox counter range (offset high word = rank)."""
    return rank << 32


# --------------------------------------------------------------------------------------------
# Bytes
# --------------------------------------------------------------------------------------------
def chain_bytes(B, k, V, esize, with_q=False):
    logits = B * (k + 1) * V * esize
    q = B * k * V * 4 if with_q else 0
    return logits + q + B * k * 4 + B * (k + 1) * 4 + B * 4


def tree_bytes(B, N, V, esize):
    return B * N * V * esize + 2 * B * N * 4 + 2 * B * N * 4 + B * 4


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


# --------------------------------------------------------------------------------------------
# Clock sampling during the timed region
# --------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            if t0 - 0.05 <= ts <= t1 + 0.05:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[4:8]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((num(r[2]) or 0.0) for r in rows)}


def gpu_selector(torch, dev) -> str:
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        return uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        return str(dev.index or 0)


def capture_calls(torch, calls):
    """One CUDA graph holding the given launches back to back (each call enqueues on the current
    stream, which is the capture stream inside the block)."""
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls[0]()  # warm-up outside capture on the side stream (first-use setup, if any)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        for c in calls:
            c()
    return graph


def graph_time_ms(torch, calls, reps, flush=None):
    """Per-call device time (ms) of calls replayed back to back from one CUDA graph."""
    graph = capture_calls(torch, calls)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * len(calls))
    # Flushed: one call per graph, L2 cleared between replays, each replay timed on its own.
    times = []
    for _ in range(reps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times) / len(calls)


# --------------------------------------------------------------------------------------------
# Our arm
# --------------------------------------------------------------------------------------------
def run_ours(args, D: Dist):
    import numpy as np
    import torch

    import speculative_decoding_verification_verify_gb300 as sv
    from speculative_decoding_verification_verify_gb300 import binding
    from speculative_decoding_verification_verify_gb300 import workloads as wl

    dev = torch.device("cuda", D.local_rank)
    torch.cuda.set_device(dev)
    D.init("nccl")
    lib = sv.load_library()
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    off0 = rank_offset(D.rank)

    # Inputs: N_SETS independent batches, resident in HBM.
    sets = []
    ws_bytes = sv.spec_verify_workspace_bytes(sv.MODE_REJECTION, B, K_DRAFTS, V)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for i in range(N_SETS):
        inp = wl.chain_b64k7(dev, seed=1236 + 101 * i + 7919 * D.rank)
        out = torch.empty((B, K_DRAFTS + 1), dtype=torch.int32, device=dev)
        alen = torch.empty(B, dtype=torch.int32, device=dev)
        sets.append((inp, out, alen))
    torch.cuda.synchronize()

    def call(i, offset):
        inp, out, alen = sets[i % N_SETS]
        rc = lib.spec_verify_rejection(
            ctypes.c_void_p(inp.logits.data_ptr()), sv.BF16, ctypes.c_void_p(inp.drafts.data_ptr()),
            None, B, K_DRAFTS, V, 1.0, inp.seed, offset, ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(alen.data_ptr()), None, ctypes.c_void_p(ws.data_ptr()), ws_bytes,
            ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        if rc != 0:
            raise RuntimeError(f"spec_verify_rejection returned {rc}")

    for w in range(args.warmup):
        call(w, off0 + w)
    torch.cuda.synchronize()

    # The timed region replays a CUDA graph of GRAPH_CALLS back-to-back calls (the input sets
    # rotate, each call has its own Philox offset), so host launch overhead does not pace the GPU.
    graph = capture_calls(torch, [lambda i=i: call(i, off0 + args.warmup + i) for i in range(GRAPH_CALLS)])
    reps = max(1, args.steps // GRAPH_CALLS)
    K = reps * GRAPH_CALLS
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_selector(torch, dev))
    time.sleep(0.1)
    D.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    # One event pair per replay (30 calls each) gives the spread; their span gives the total.
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record()
    for i in range(reps):
        graph.replay()
        ev[i + 1].record()
    torch.cuda.synchronize()
    t1 = time.time()
    D.barrier()
    clocks.stop()
    total_ms = ev[0].elapsed_time(ev[-1])
    per_call = [ev[i].elapsed_time(ev[i + 1]) / GRAPH_CALLS for i in range(reps)]
    launch_ms = total_ms / K
    max_total_ms = D.max(total_ms, dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during the benchmark")

    positions = B * (K_DRAFTS + 1)
    value = D.world * positions * K / (max_total_ms * 1e-3)
    alg = chain_bytes(B, K_DRAFTS, V, 2)
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_kind = "measured" if peak else "fallback"
    if not peak:
        peak = 6800.0
    achieved = alg / (launch_ms * 1e-3) / 1e9
    traffic = None
    try:
        tr = json.load(open(PROFILE_TRAFFIC))
        if tr.get("kernel_source_hash") == kernel_source_hash():
            traffic = tr.get("dram_bytes_per_call")
    except (OSError, ValueError):
        pass

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": D.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": max_total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "k": K_DRAFTS, "V": V, "logits": "bf16",
                   "mode": "target-only (one-hot q)", "positions_per_step": positions,
                   "l2": f"{N_SETS} rotating input sets of {alg / 1e6:.1f} MB each (> L2)"},
        # The timed unit is one whole verify call: the streaming kernel and the finaliser it
        # launches as a programmatic dependent.  Events between the two would serialise them,
        # so the streaming kernel alone is not timed here; its share of the call is in the ncu
        # launch list under profiles/.
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": alg,
                     "kernel": "verify call: sv_stream_kernel<bf16, sample> + sv_finalize_kernel<bf16, sample>",
                     "launch_ms": launch_ms,
                     "launch_ms_median_p10_p90": [statistics.median(per_call),
                                                  float(np.percentile(per_call, 10)),
                                                  float(np.percentile(per_call, 90))],
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "timing": f"CUDA events around each of {reps} replays of a graph of {GRAPH_CALLS} calls"},
        "gpu_launches": LAUNCHES_PER_CALL * K,
        "clocks": clocks.summary(t0, t1),
    }

    # End to end through the same C ABI with host buffers: H2D of the step's inputs from pinned
    # memory, the call, D2H of its outputs, every step.
    if not args.no_e2e:
        line["e2e"] = run_e2e(args, D, torch, sv, lib, sets, ws, ws_bytes, status, stream, sh, off0)

    if D.rank == 0 and D.world == 1 and args.cpu_seconds > 0:
        line["cpu_baseline"] = cpu_baseline(sets[0][0], args.cpu_seconds)
    if not args.no_modes:
        line["modes"] = other_modes(args, D, torch, sv, wl, dev, stream, peak)
    D.close()
    if D.rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, D, torch, sv, lib, sets, ws, ws_bytes, status, stream, sh, off0):
    """End to end through the C ABI from pinned host buffers: every step copies its logits and
    drafts host -> device, verifies, and copies the outputs back.  The device inputs are double
    buffered: step s + 1's copy (on a copy stream) overlaps step s's verification, which is
    what a serving loop does; the host -> device link (about 210 GB/s on this machine) bounds
    the rate."""
    steps = min(args.steps, 200)
    host = []
    for inp, out, alen in sets[:2]:
        hl = torch.empty(inp.logits.shape, dtype=inp.logits.dtype, pin_memory=True)
        hl.copy_(inp.logits)
        hd = torch.empty(inp.drafts.shape, dtype=torch.int32, pin_memory=True)
        hd.copy_(inp.drafts)
        ho = torch.empty(sets[0][1].shape, dtype=torch.int32, pin_memory=True)
        ha = torch.empty(sets[0][2].shape, dtype=torch.int32, pin_memory=True)
        host.append((hl, hd, ho, ha, inp.seed))
    dev_in = [(torch.empty_like(sets[0][0].logits), torch.empty_like(sets[0][0].drafts)) for _ in range(2)]
    out, alen = sets[0][1], sets[0][2]
    h2d = sets[0][0].logits.numel() * sets[0][0].logits.element_size() + sets[0][0].drafts.numel() * 4
    d2h = out.numel() * 4 + alen.numel() * 4
    copy_stream = torch.cuda.Stream(device=stream.device)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def issue_copy(s):
        hl, hd = host[s % len(host)][:2]
        dl, dd = dev_in[s % 2]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[s % 2])  # the step that last read this buffer is done
            dl.copy_(hl, non_blocking=True)
            dd.copy_(hd, non_blocking=True)
            copied[s % 2].record(copy_stream)

    def verify(s, offset):
        _, _, ho, ha, seed = host[s % len(host)]
        dl, dd = dev_in[s % 2]
        stream.wait_event(copied[s % 2])
        rc = lib.spec_verify_rejection(
            ctypes.c_void_p(dl.data_ptr()), sv.BF16, ctypes.c_void_p(dd.data_ptr()), None, B,
            K_DRAFTS, V, 1.0, seed, offset, ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(alen.data_ptr()), None, ctypes.c_void_p(ws.data_ptr()), ws_bytes,
            ctypes.c_void_p(status.data_ptr()), sh)
        consumed[s % 2].record(stream)
        ho.copy_(out, non_blocking=True)
        ha.copy_(alen, non_blocking=True)
        return rc

    def run(n, base):
        issue_copy(0)
        for s in range(n):
            if s + 1 < n:
                issue_copy(s + 1)
            assert verify(s, base + s) == 0

    for e in consumed:
        e.record(stream)
    run(3, off0 + 10**6)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    D.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    copy_stream.wait_event(e0)
    run(steps, off0 + 2 * 10**6)
    e1.record(stream)
    torch.cuda.synchronize()
    D.barrier()
    ms = D.max(e0.elapsed_time(e1), torch.device("cuda", D.local_rank))
    return {"value": D.world * B * (K_DRAFTS + 1) * steps / (ms * 1e-3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms / steps, "gpu_launches": LAUNCHES_PER_CALL * steps,
            "h2d_gbs": h2d * steps / (ms * 1e-3) / 1e9,
            "path": "pinned host -> device copy (double-buffered, copy stream), spec_verify_rejection, "
                    "device -> pinned host"}


def _oracle_rate(lg, d, seed, seconds, threads):
    """Requests of the workload verified per second by the oracle on `threads` host threads
    (each thread verifies whole requests; the oracle's C code runs without the GIL)."""
    import concurrent.futures as cf

    import numpy as np

    import oracle

    stop = time.perf_counter() + seconds
    counter = iter(range(1 << 30))

    def worker():
        n = 0
        while time.perf_counter() < stop or n == 0:
            b = next(counter) % B
            oracle.verify_rejection(lg, d, None, 1.0, seed, 0, req_ids=np.array([b], np.int32))
            n += 1
        return n

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        done = sum(ex.map(lambda _: worker(), range(threads)))
    el = time.perf_counter() - t0
    return done, el


def cpu_baseline(inp, seconds):
    from speculative_decoding_verification_verify_gb300 import workloads as wl

    import oracle

    lg = wl.to_numpy_logits(inp.logits)
    d = inp.drafts.cpu().numpy()
    oracle.build()
    threads = os.cpu_count() or 1
    n1, el1 = _oracle_rate(lg, d, inp.seed, seconds / 2, 1)
    nt, elt = _oracle_rate(lg, d, inp.seed, seconds / 2, threads)
    return {"value": nt * (K_DRAFTS + 1) / elt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{nt} requests (8 positions each) of the b64k7 workload on {threads} threads, "
                      f"{elt:.1f} s",
            "single_thread": {"value": n1 * (K_DRAFTS + 1) / el1, "cores": 1,
                              "sample": f"{n1} requests, {el1:.1f} s"}}


# --------------------------------------------------------------------------------------------
# The other modes, timed briefly (per-launch CUDA events, L2 handled per workload)
# --------------------------------------------------------------------------------------------
def other_modes(args, D, torch, sv, wl, dev, stream, peak):
    """The other verify modes through the C ABI, preallocated buffers, CUDA-graph replays."""
    lib = sv.load_library()
    P = lambda t: ctypes.c_void_p(None if t is None else t.data_ptr())
    cur = lambda: ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def check(rc, name):
        if rc != 0:
            raise RuntimeError(f"{name} returned {rc}")

    res = {}
    names = {"greedy", "tree", "block", "with_q", "b1k3", "kv_compact", "variants", "budget"}
    want = names if args.modes == "all" else set(args.modes.split(","))
    if want - names:
        raise SystemExit(f"unknown modes {sorted(want - names)}; known: {sorted(names)}")
    out = torch.empty((B, K_DRAFTS + 1), dtype=torch.int32, device=dev)
    alen = torch.empty(B, dtype=torch.int32, device=dev)
    if "greedy" in want:
        res.update(_greedy_mode(torch, sv, wl, dev, lib, P, cur, check, status, out, alen, peak))
    if "tree" in want:
        res.update(_tree_modes(torch, sv, wl, dev, lib, P, cur, check, status, peak))
    if want & {"block", "with_q"}:
        res.update(_block_modes(torch, sv, wl, dev, lib, P, cur, check, status, out, alen, peak, want))
    if "b1k3" in want:
        res.update(_b1k3_mode(torch, sv, wl, dev, lib, P, cur, check, status, peak))
    if "variants" in want:
        res.update(_variant_modes(torch, sv, wl, dev, lib, P, cur, check, status, out, alen, peak))
    if "budget" in want:
        res.update(_budget_modes(torch, sv, dev, lib, P, cur, check))
    if "kv_compact" in want:
        res.update(_kv_mode(torch, wl, dev, lib, P, cur, check, status, peak, args.kv_max_pos))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the other modes")
    return res


def _greedy_mode(torch, sv, wl, dev, lib, P, cur, check, status, out, alen, peak):
    """Greedy on the headline workload (3 rotating sets > L2)."""
    sets = [wl.chain_b64k7(dev, seed=5000 + i) for i in range(N_SETS)]
    nb = sv.spec_verify_workspace_bytes(sv.MODE_GREEDY, B, K_DRAFTS, V)
    ws = torch.zeros(nb, dtype=torch.uint8, device=dev)

    def greedy(i):
        x = sets[i % N_SETS]
        check(lib.spec_verify_greedy(P(x.logits), sv.BF16, P(x.drafts), B, K_DRAFTS, V, P(out), P(alen),
                                     P(ws), nb, P(status), cur()), "spec_verify_greedy")

    ms = graph_time_ms(torch, [lambda i=i: greedy(i) for i in range(GRAPH_CALLS)], 20)
    return {"greedy_b64k7": _mode_entry(ms, B * (K_DRAFTS + 1), chain_bytes(B, K_DRAFTS, V, 2), peak, 2)}


def _tree_modes(torch, sv, wl, dev, lib, P, cur, check, status, peak):
    """Tree, both modes (3 x 117 MB)."""
    res = {}
    trees = [wl.tree_b48(dev, seed=6000 + i) for i in range(N_SETS)]
    Bt, Nt, Vt = trees[0].shape
    tout = torch.empty((Bt, Nt), dtype=torch.int32, device=dev)
    tai = torch.empty((Bt, Nt), dtype=torch.int32, device=dev)
    tal = torch.empty(Bt, dtype=torch.int32, device=dev)
    nb = sv.spec_verify_workspace_bytes(sv.MODE_TREE, Bt, Nt, Vt)
    tws = torch.zeros(nb, dtype=torch.uint8, device=dev)
    for mode, name in ((0, "tree_b48_greedy"), (1, "tree_b48_target_only")):
        def tree(i, mode=mode):
            x = trees[i % N_SETS]
            check(lib.spec_verify_tree(P(x.logits), sv.BF16, P(x.node_tokens), P(x.parents), Bt, Nt, Vt, mode,
                                       1.0, 1, i, P(tout), P(tai), P(tal), P(tws), nb, P(status), cur()),
                  "spec_verify_tree")

        ms = graph_time_ms(torch, [lambda i=i: tree(i) for i in range(GRAPH_CALLS)], 20)
        res[name] = _mode_entry(ms, Bt * Nt, tree_bytes(Bt, Nt, Vt, 2), peak, 2)
    return res


def _block_modes(torch, sv, wl, dev, lib, P, cur, check, status, out, alen, peak, want):
    """Block verification: one-hot on the headline workload, and with draft probabilities (with
    the standard rule beside it) on the sweep's B=64, k=7 cell (logits 131 MB + q 230 MB per
    call, 3 sets)."""
    res = {}
    nb = sv.spec_verify_workspace_bytes(sv.MODE_BLOCK, B, K_DRAFTS, V)
    bws = torch.zeros(nb, dtype=torch.uint8, device=dev)

    def block(i, x, q):
        check(lib.spec_verify_block(P(x.logits), sv.BF16, P(x.drafts), P(q), B, K_DRAFTS, V, 1.0, x.seed, i,
                                    P(out), P(alen), P(bws), nb, P(status), cur()), "spec_verify_block")

    if "block" in want:
        sets = [wl.chain_b64k7(dev, seed=7000 + i) for i in range(N_SETS)]
        ms = graph_time_ms(torch, [lambda i=i: block(i, sets[i % N_SETS], None) for i in range(GRAPH_CALLS)], 20)
        res["block_b64k7_one_hot"] = _mode_entry(ms, B * (K_DRAFTS + 1), chain_bytes(B, K_DRAFTS, V, 2), peak, 2)
        del sets
    if "with_q" not in want:
        return res
    qsets = [wl.chain_sweep(dev, seed=7100 + i, B=B, k=K_DRAFTS, alpha=0.7) for i in range(N_SETS)]
    ms = graph_time_ms(torch, [lambda i=i: block(i, qsets[i % N_SETS], qsets[i % N_SETS].q) for i in range(12)], 10)
    nr = sv.spec_verify_workspace_bytes(sv.MODE_REJECTION, B, K_DRAFTS, V)
    rws = torch.zeros(nr, dtype=torch.uint8, device=dev)

    def standard_q(i, x):
        check(lib.spec_verify_rejection(P(x.logits), sv.BF16, P(x.drafts), P(x.q), B, K_DRAFTS, V, 1.0, x.seed, i,
                                        P(out), P(alen), None, P(rws), nr, P(status), cur()), "spec_verify_rejection")

    sms = graph_time_ms(torch, [lambda i=i: standard_q(i, qsets[i % N_SETS]) for i in range(12)], 10)
    res["standard_sweep_b64k7_with_q"] = _mode_entry(
        sms, B * (K_DRAFTS + 1), chain_bytes(B, K_DRAFTS, V, 2, with_q=True), peak, 3,
        note="algorithmic bytes count all of q; the residual kernel reads q only at rejected rows")
    res["block_sweep_b64k7_with_q"] = _mode_entry(
        ms, B * (K_DRAFTS + 1), chain_bytes(B, K_DRAFTS, V, 2, with_q=True), peak, 3,
        note="algorithmic bytes count the logits and q once; the block kernel reads the logits and q "
             "of the present rows a second time")
    del qsets
    return res


def _b1k3_mode(torch, sv, wl, dev, lib, P, cur, check, status, peak):
    """Standard rejection, B=1 k=3 (2.6 MB: L2 flushed before each call)."""
    inp = wl.chain_b1k3(dev)
    Bq, kq, Vq = inp.shape
    qout = torch.empty((Bq, kq + 1), dtype=torch.int32, device=dev)
    qal = torch.empty(Bq, dtype=torch.int32, device=dev)
    nb = sv.spec_verify_workspace_bytes(sv.MODE_REJECTION, Bq, kq, Vq)
    qws = torch.zeros(nb, dtype=torch.uint8, device=dev)
    flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def standard():
        check(lib.spec_verify_rejection(P(inp.logits), sv.BF16, P(inp.drafts), P(inp.q), Bq, kq, Vq,
                                        inp.temperature, inp.seed, 7, P(qout), P(qal), None, P(qws), nb,
                                        P(status), cur()), "spec_verify_rejection")

    ms = graph_time_ms(torch, [standard], 100, flush=lambda: flush_buf.zero_())
    return {"standard_b1k3": _mode_entry(ms, Bq * (kq + 1), chain_bytes(Bq, kq, Vq, 2, with_q=True),
                                         peak, 3, note="latency-bound; L2 flushed before each call; "
                                         "algorithmic bytes count all of q")}


def _variant_modes(torch, sv, wl, dev, lib, P, cur, check, status, out, alen, peak):
    """Verify variants on the headline workload: a temperature per request (every other request
    greedy, the rest sampling at T in [0.6, 1.4]), relaxed thresholds (0.5, 0.5), and top-k 50 with
    top-p 0.9 on every request."""
    import ctypes as ct

    res = {}
    sets = [wl.chain_b64k7(dev, seed=9000 + i) for i in range(N_SETS)]
    nb = sv.spec_verify_workspace_bytes(sv.MODE_REJECTION, B, K_DRAFTS, V)
    ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
    temps = torch.linspace(0.6, 1.4, B, device=dev)
    temps[::2] = 0.0
    top_k = torch.full((B,), 50, dtype=torch.int32, device=dev)
    top_p = torch.full((B,), 0.9, dtype=torch.float32, device=dev)
    opts = {"mixed_temperatures_b64k7": sv.Options(temps.data_ptr(), 1.0, 1.0, 1.0, None, None),
            "relaxed_thresholds_b64k7": sv.Options(None, 1.0, 0.5, 0.5, None, None),
            "top_k50_top_p0.9_b64k7": sv.Options(None, 1.0, 1.0, 1.0, top_k.data_ptr(), top_p.data_ptr())}
    for name, opt in opts.items():
        def call(i, opt=opt):
            x = sets[i % N_SETS]
            check(lib.spec_verify_rejection_ex(P(x.logits), sv.BF16, P(x.drafts), None, B, K_DRAFTS, V,
                                               ct.byref(opt), x.seed, i, P(out), P(alen), None, P(ws), nb,
                                               P(status), cur()), "spec_verify_rejection_ex")

        ms = graph_time_ms(torch, [lambda i=i: call(i) for i in range(GRAPH_CALLS)], 20)
        launches = 3 if name.startswith("top_k") else 2
        res[name] = _mode_entry(ms, B * (K_DRAFTS + 1), chain_bytes(B, K_DRAFTS, V, 2), peak, launches,
                                note="the threshold kernel reads each row several times" if launches == 3 else None)
    return res


def _budget_modes(torch, sv, dev, lib, P, cur, check):
    """The adaptive verification budget (keys, rank, pick) on B x K slots of random confidences
    with a roofline-shaped cost table; latency per plan."""
    res = {}
    g = torch.Generator(device=dev).manual_seed(5)
    for B_, K_ in ((512, 7), (2048, 8)):
        conf = torch.rand((B_, K_), generator=g, device=dev) * 0.5 + 0.5
        b = torch.arange(B_ * K_ + 1, device=dev, dtype=torch.float64)
        cost = 1.25e-3 + torch.clamp((B_ + b) * 3e-5 - 1e-3, min=0.0)
        adm = torch.empty(B_, dtype=torch.int32, device=dev)
        bud = torch.empty(1, dtype=torch.int32, device=dev)

        nws = int(lib.spec_verify_plan_budget_workspace_bytes(B_, K_))
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)

        def plan():
            check(lib.spec_verify_plan_budget(P(conf), None, B_, K_, P(cost), P(adm), P(bud), None, P(ws), nws,
                                              cur()), "spec_verify_plan_budget")

        ms = graph_time_ms(torch, [plan] * 10, 20)
        res[f"plan_budget_B{B_}_K{K_}"] = {"ms_per_call": ms, "slots": B_ * K_, "budget": int(bud.item()),
                                          "launches_per_call": 4,
                                          "note": "latency-bound: keys, a GPU-wide rank, scatter, one picking CTA"}
    return res


def _kv_mode(torch, wl, dev, lib, P, cur, check, status, peak, max_pos):
    """KV compaction after tree verification: a Llama-3-8B-sized cache (64 planes of 2048-byte
    rows; 3.2 GB at 512 positions a request), B=48 requests of N=8 nodes; KV_SETS index sets over
    the one pool, so the rows a call moves (about 9 MB) are not in L2 from the last call that
    touched them."""
    res = {}
    kvs = [wl.kv_paged(dev, seed=8000, max_pos=max_pos)]
    for i in range(1, KV_SETS):
        kvs.append(wl.kv_paged(dev, seed=8000 + i, max_pos=max_pos, pool=kvs[0].pool))
    pool = kvs[0].pool
    planes, num_slots, row_el = pool.shape
    row_bytes = row_el * pool.element_size()
    Bk, Nk = kvs[0].accept_index.shape
    c_out = torch.empty(Bk, dtype=torch.int32, device=dev)
    moved = 0
    for x in kvs:
        ai, al = x.accept_index.cpu(), x.accept_len.cpu()
        moved += sum(int((ai[b, 1:int(al[b]) + 1] != torch.arange(1, int(al[b]) + 1)).sum()) for b in range(Bk))

    def kv(i):
        x = kvs[i]
        check(lib.spec_verify_kv_compact(P(pool), num_slots, row_bytes, planes, pool.stride(0) * pool.element_size(),
                                         P(x.slot_table), x.slot_table.shape[1], P(x.committed), P(c_out),
                                         P(x.accept_index), P(x.accept_len), Bk, Nk, P(status), cur()),
              "spec_verify_kv_compact")

    ms = graph_time_ms(torch, [lambda i=i: kv(i) for i in range(KV_SETS)], 20)
    alg = (2 * moved * planes * row_bytes) / KV_SETS + Bk * (Nk * 4 + 12 + 2 * (Nk + 1) * 4)
    e = _mode_entry(ms, Bk * Nk, alg, peak, 1,
                    note="rows_moved_per_call counts accepted-path rows whose slot changes; algorithmic "
                         "bytes = read + write of those rows in every plane, plus the index reads")
    e["rows_moved_per_call"] = moved / KV_SETS
    e["planes"], e["row_bytes"], e["max_pos"] = int(planes), int(row_bytes), int(max_pos)
    res["kv_compact_b48_llama8b"] = e
    return res


def _mode_entry(ms, positions, alg, peak, launches, note=None):
    gbs = alg / (ms * 1e-3) / 1e9
    e = {"ms_per_call": ms, "positions_per_s": positions / (ms * 1e-3),
         "algorithmic_bytes": alg, "gbs": gbs, "frac_of_peak": gbs / peak,
         "launches_per_call": launches}
    if note:
        e["note"] = note
    return e


# --------------------------------------------------------------------------------------------
# Reference arm: the CPU oracle on the same workload
# --------------------------------------------------------------------------------------------
def run_reference(args, D: Dist):
    if D.rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    from speculative_decoding_verification_verify_gb300 import workloads as wl

    oracle.build()
    inp = wl.chain_b64k7("cpu", seed=1236)
    lg = wl.to_numpy_logits(inp.logits)
    d = inp.drafts.numpy()

    import concurrent.futures as cf

    threads = os.cpu_count() or 1
    pool = cf.ThreadPoolExecutor(max_workers=threads)

    def step(s):
        # One step verifies `threads` requests of the workload, one per host thread.
        ids = [(s * threads + i) % B for i in range(threads)]
        list(pool.map(lambda b: oracle.verify_rejection(lg, d, None, 1.0, inp.seed, s,
                                                        req_ids=np.array([b], np.int32)), ids))

    for w in range(args.warmup):
        step(w)
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(args.warmup + s)
    el = time.perf_counter() - t0
    pool.shutdown()
    value = (K_DRAFTS + 1) * threads * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": D.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "k": K_DRAFTS, "V": V, "logits": "bf16",
                   "mode": "target-only (one-hot q)",
                   "step": f"{threads} requests (8 positions each) of the workload per step, one per host thread"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} steps of {threads} requests of the b64k7 workload"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    del torch


def main():
    args = parse_args()
    D = Dist()
    if args.impl == "reference":
        run_reference(args, D)
    else:
        run_ours(args, D)


if __name__ == "__main__":
    main()
