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
import contextlib
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
GRAPH_CALLS = 30  # verify calls captured in one CUDA graph when timing the other modes
MAX_GRAPH_CALLS = 100  # largest graph of headline calls; more steps replay it several times
SPREAD_REPLAYS = 10   # replays, after the timed region, that give the per-call spread
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


@contextlib.contextmanager
def nvtx_range(torch, name):
    """A named NVTX range around a phase of the bench (seen by Nsight tools; a no-op without one)."""
    pushed = False
    try:
        torch.cuda.nvtx.range_push(name)
        pushed = True
    except Exception:
        pass
    try:
        yield
    finally:
        if pushed:
            torch.cuda.nvtx.range_pop()


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work spent timing the oracle baseline")
    ap.add_argument("--no-modes", action="store_true", help="skip the other verify modes")
    ap.add_argument("--budget-shapes", default="512x7,2048x8",
                    help="B x K shapes of the budget mode, comma-separated (default 512x7,2048x8)")
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


def required_bytes(B, k, V, esize, rejected_rows):
    """Bytes standard rejection must read: every logit once, q at each draft (a gather), one q row
    per request whose round stops at a rejected draft (the residual max(0, p - q) needs that whole
    row), the drafts, and the outputs."""
    return B * (k + 1) * V * esize + B * k * 4 + rejected_rows * V * 4 + B * k * 4 + B * (k + 1) * 4 + B * 4


def rejected_rows(alen, k, drafts):
    """Requests whose round stopped at a present draft (a rejection, not a bonus or a gap)."""
    a = alen.cpu().numpy()
    d = drafts.cpu().numpy()
    return int(sum(1 for b in range(a.shape[0]) if 0 <= a[b] < k and d[b, a[b]] >= 0))


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


def _event(torch):
    """A timing event that can be recorded inside a CUDA graph (an event-record node)."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:  # a torch without external events: record around the replay instead
        return None


class TimedGraph:
    """One CUDA graph holding the given calls back to back (each enqueues on the current stream,
    the capture stream inside the block), bracketed by two timing events recorded inside the graph
    where torch supports it, so a replay's interval is the device time of exactly these calls."""

    def __init__(self, torch, calls):
        self.torch = torch
        self.n = len(calls)
        self.graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            calls[0]()  # first-use setup, if any, outside capture
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.e0, self.e1 = _event(torch), _event(torch)
        self.inside = self.e0 is not None and self.e1 is not None
        if not self.inside:
            self.e0 = torch.cuda.Event(enable_timing=True)
            self.e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.graph(self.graph):
            if self.inside:
                self.e0.record()
            for c in calls:
                c()
            if self.inside:
                self.e1.record()

    def replay(self):
        if not self.inside:
            self.e0.record()
        self.graph.replay()
        if not self.inside:
            self.e1.record()

    def last_ms(self):
        """Device time of the last replay (call after synchronising)."""
        return self.e0.elapsed_time(self.e1)


def graph_time_ms(torch, calls, reps, flush=None):
    """Per-call device time (ms): median over `reps` replays of a graph of the calls.  With
    `flush` the graph holds one call and the flush runs before each replay, outside the timed
    interval."""
    tg = TimedGraph(torch, calls)
    for _ in range(3):
        if flush is not None:
            flush()
        tg.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        if flush is not None:
            flush()
        tg.replay()
        torch.cuda.synchronize()
        times.append(tg.last_ms() / tg.n)
    return statistics.median(times)


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

    with nvtx_range(torch, "warmup"):
        for w in range(args.warmup):
            call(w, off0 + w)
        torch.cuda.synchronize()

    # The timed region is exactly K calls (the input sets rotate, each call has its own Philox
    # offset), replayed from CUDA graphs so that host launches do not pace the GPU: one graph of
    # all K calls when K <= MAX_GRAPH_CALLS (its timing events recorded inside the graph), else
    # graphs of MAX_GRAPH_CALLS calls and one of the remainder, replayed back to back.
    K = args.steps
    base = off0 + args.warmup
    GC = min(K, MAX_GRAPH_CALLS)
    nfull, rem = divmod(K, GC)
    main = TimedGraph(torch, [lambda i=i: call(i, base + i) for i in range(GC)])
    tail = (TimedGraph(torch, [lambda i=i: call(nfull * GC + i, base + nfull * GC + i) for i in range(rem)])
            if rem else None)
    for _ in range(3):
        main.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_selector(torch, dev))
    time.sleep(0.1)
    # One more untimed replay right before the timed region: the pause above (the clock sampler
    # starting) lets the GPU drop out of its busy state, which the first replay after it pays for.
    main.replay()
    torch.cuda.synchronize()
    D.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with nvtx_range(torch, "timed region"):
        if nfull == 1 and tail is None:
            main.replay()
            torch.cuda.synchronize()
            total_ms = main.last_ms()
        else:
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            for _ in range(nfull):
                main.replay()
            if tail is not None:
                tail.replay()
            s1.record()
            torch.cuda.synchronize()
            total_ms = s0.elapsed_time(s1)
    t1 = time.time()
    D.barrier()
    clocks.stop()
    launch_ms = total_ms / K
    max_total_ms = D.max(total_ms, dev)
    # The spread, outside the timed region: per-call time over further replays of the graph.
    per_call = []
    with nvtx_range(torch, "spread replays"):
        for _ in range(SPREAD_REPLAYS):
            main.replay()
            torch.cuda.synchronize()
            per_call.append(main.last_ms() / main.n)
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
                     "timing": (f"{K} calls from CUDA graphs of {GC} calls"
                                + (", timing events recorded inside the graph" if main.inside else "")
                                + f"; spread over {SPREAD_REPLAYS} further replays of {GC} calls")},
        "gpu_launches": LAUNCHES_PER_CALL * K,
        "clocks": clocks.summary(t0, t1),
    }

    # End to end through the same C ABI with host buffers: H2D of the step's inputs from pinned
    # memory, the call, D2H of its outputs, every step.
    if not args.no_e2e:
        with nvtx_range(torch, "end to end"):
            line["e2e"] = run_e2e(args, D, torch, sv, lib, sets, ws, ws_bytes, status, stream, sh, off0)

    if D.rank == 0:
        with nvtx_range(torch, "acceptance"):
            line["acceptance"] = acceptance_stats(lib, sv, torch, sets[0], ws, ws_bytes, off0 + 12345)
    if D.rank == 0 and D.world == 1 and args.cpu_seconds > 0:
        line["cpu_baseline"] = cpu_baseline(sets[0][0], args.cpu_seconds)
    if not args.no_modes:
        with nvtx_range(torch, "other modes"):
            line["modes"] = other_modes(args, D, torch, sv, wl, dev, stream, peak)
    D.close()
    if D.rank == 0:
        print(json.dumps(line), flush=True)


def gpu_numa_node(torch, dev):
    """The NUMA node the GPU's PCI function reports (sysfs), or None."""
    try:
        pr = torch.cuda.get_device_properties(dev)
        bus = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        node = int(open(f"/sys/bus/pci/devices/{bus}/numa_node").read().strip())
        return node if node >= 0 else None
    except (AttributeError, OSError, ValueError):
        return None


def node_cpus(node):
    """CPUs of a NUMA node (sysfs cpulist), or an empty set."""
    try:
        txt = open(f"/sys/devices/system/node/node{node}/cpulist").read().strip()
    except OSError:
        return set()
    cpus = set()
    for part in txt.split(","):
        if "-" in part:
            lo, hi = part.split("-")
            cpus.update(range(int(lo), int(hi) + 1))
        elif part:
            cpus.add(int(part))
    return cpus


class NodeBinding:
    """Bind this thread's CPU affinity and memory policy to one NUMA node while pinned host
    buffers are allocated and the end-to-end leg runs (process settings only; no GPU setting is
    touched).  Restores both on exit."""
    MPOL_DEFAULT, MPOL_BIND = 0, 2
    NR_SET_MEMPOLICY = {"aarch64": 237, "x86_64": 238}

    def __init__(self, node):
        self.node, self.ok, self.mem_ok = node, False, False
        self.old_aff = None

    def _set_mempolicy(self, mode, mask):
        import platform

        nr = self.NR_SET_MEMPOLICY.get(platform.machine())
        if nr is None:
            return False
        libc = ctypes.CDLL(None, use_errno=True)
        m = ctypes.c_ulong(mask)
        return libc.syscall(nr, mode, ctypes.byref(m) if mask else None, 64 if mask else 0) == 0

    def __enter__(self):
        cpus = node_cpus(self.node) if self.node is not None else set()
        if cpus:
            self.old_aff = os.sched_getaffinity(0)
            os.sched_setaffinity(0, cpus)
            self.ok = True
            self.mem_ok = self._set_mempolicy(self.MPOL_BIND, 1 << self.node)
        return self

    def __exit__(self, *exc):
        if self.mem_ok:
            self._set_mempolicy(self.MPOL_DEFAULT, 0)
        if self.old_aff is not None:
            os.sched_setaffinity(0, self.old_aff)


def run_e2e(args, D, torch, sv, lib, sets, ws, ws_bytes, status, stream, sh, off0):
    """End to end through the C ABI from pinned host buffers: every step copies its logits and
    drafts host -> device, verifies, and copies the outputs back.  The device inputs are double
    buffered: step s + 1's copy (on a copy stream) overlaps step s's verification, which is what a
    serving loop does; the host -> device link bounds the rate.  Measured with the process as it
    starts, and again with its CPU affinity and memory policy bound to the GPU's NUMA node (the
    pinned buffers allocated under that policy); the line reports the bound run when the node is
    known."""
    node = gpu_numa_node(torch, stream.device)
    plain = _e2e_once(args, D, torch, sv, lib, sets, ws, ws_bytes, status, stream, sh, off0)
    plain["numa"] = {"gpu_node": node, "bound": False}
    if node is None:
        return plain
    with NodeBinding(node) as nb:
        if not nb.ok:
            return plain
        bound = _e2e_once(args, D, torch, sv, lib, sets, ws, ws_bytes, status, stream, sh, off0)
    bound["numa"] = {"gpu_node": node, "bound": True, "memory_policy_bound": nb.mem_ok,
                     "cpus": len(node_cpus(node))}
    bound["unbound"] = {k: plain[k] for k in ("value", "ms_per_step", "h2d_gbs")}
    return bound


def _e2e_once(args, D, torch, sv, lib, sets, ws, ws_bytes, status, stream, sh, off0):
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
    del host, hl, hd, ho, ha
    # Pinned blocks go back to torch's host cache; empty it so the next leg allocates afresh
    # (under its own memory policy).
    if hasattr(torch._C, "_host_emptyCache"):
        torch._C._host_emptyCache()
    return {"value": D.world * B * (K_DRAFTS + 1) * steps / (ms * 1e-3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms / steps, "gpu_launches": LAUNCHES_PER_CALL * steps,
            "h2d_gbs": h2d * steps / (ms * 1e-3) / 1e9,
            "path": "pinned host -> device copy (double-buffered, copy stream), spec_verify_rejection, "
                    "device -> pinned host"}


def acceptance_stats(lib, sv, torch, one_set, ws, ws_bytes, offset):
    """What the round emitted on the timed batch (input set 0, one Philox offset), outside the
    timed region: the oracle's accepted lengths, the accepted-per-position counts (requests whose
    draft at position i was accepted), the emitted tokens per request, and the draws the oracle
    flags as lying within 1e-6 of a decision boundary; the GPU's outputs of the same call are
    compared with the oracle's request by request."""
    import numpy as np

    import oracle
    from speculative_decoding_verification_verify_gb300 import workloads as wl

    inp, out, alen = one_set
    st = torch.zeros(1, dtype=torch.int32, device=out.device)
    rc = lib.spec_verify_rejection(
        ctypes.c_void_p(inp.logits.data_ptr()), sv.BF16, ctypes.c_void_p(inp.drafts.data_ptr()), None, B,
        K_DRAFTS, V, 1.0, inp.seed, offset, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(alen.data_ptr()),
        None, ctypes.c_void_p(ws.data_ptr()), ws_bytes, ctypes.c_void_p(st.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc != 0:
        raise RuntimeError(f"spec_verify_rejection returned {rc}")
    torch.cuda.synchronize()
    g_tok, g_len = out.cpu().numpy(), alen.cpu().numpy()
    oracle.build()
    ref = oracle.verify_rejection(wl.to_numpy_logits(inp.logits), inp.drafts.cpu().numpy(), None, 1.0, inp.seed,
                                  offset)
    flagged = ref["boundary"].astype(bool)
    same = (g_len == ref["accept_len"]) & np.all(g_tok == ref["out_tokens"], axis=1)
    L = ref["accept_len"]
    return {"requests": int(B), "boundary_draws": int(flagged.sum()),
            "differing_requests_outside_boundary": int((~same & ~flagged).sum()),
            "device_status": int(st.item()),
            "mean_accept_len": float(L.mean()), "mean_emitted_tokens": float((L + 1).mean()),
            "accept_len_histogram": np.bincount(L, minlength=K_DRAFTS + 1).tolist(),
            "accepted_per_position": [int((L > i).sum()) for i in range(K_DRAFTS)],
            "source": f"CPU oracle on input set 0 of the timed batch at Philox offset {offset}; the GPU's "
                      "outputs of the same call compared request by request"}


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
    names = {"greedy", "tree", "block", "with_q", "b1k3", "tiny", "sweep", "kv_compact", "variants", "budget"}
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
    if "tiny" in want:
        res.update(_tiny_mode(torch, sv, wl, dev, lib, P, cur, check, status))
    if "sweep" in want:
        res.update(_sweep_modes(torch, sv, wl, dev, lib, P, cur, check, status, peak))
    if "variants" in want:
        res.update(_variant_modes(torch, sv, wl, dev, lib, P, cur, check, status, out, alen, peak))
    if "budget" in want:
        shapes = [tuple(int(x) for x in t.split("x")) for t in args.budget_shapes.split(",") if t]
        res.update(_budget_modes(torch, sv, dev, lib, P, cur, check, shapes))
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
    # The block rule needs every present row's q (its residual masses r_L sum max(0, w_L p - q) over
    # the whole row), so its bytes are the logits and all of q once; the kernel reads both a second
    # time in its residual pass.
    both = chain_bytes(B, K_DRAFTS, V, 2, with_q=True)
    e = _mode_entry(ms, B * (K_DRAFTS + 1), both, peak, 3,
                    note="bytes the block rule must read: the logits and every present q row once; the "
                         "design reads both twice (the streaming pass, then the block kernel's residual pass)")
    e["gbs_counting_both_passes"] = 2 * both / (ms * 1e-3) / 1e9
    res["block_sweep_b64k7_with_q"] = e
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
    standard()
    nrej = rejected_rows(qal, kq, inp.drafts)
    e = _mode_entry(ms, Bq * (kq + 1), required_bytes(Bq, kq, Vq, 2, nrej), peak, 3,
                    note="latency-bound; L2 flushed before each call; bytes = what the rule must read")
    e["bytes_all_of_q"] = chain_bytes(Bq, kq, Vq, 2, with_q=True)
    return {"standard_b1k3": e}


def _tiny_mode(torch, sv, wl, dev, lib, P, cur, check, status):
    """The tiny configuration (B=4, k=3, V=1024, fp32): latency of standard rejection and greedy,
    L2 flushed before each call, device time of the call alone."""
    inp = wl.chain_tiny(dev)
    Bt, kt, Vt = inp.shape
    o = torch.empty((Bt, kt + 1), dtype=torch.int32, device=dev)
    al = torch.empty(Bt, dtype=torch.int32, device=dev)
    nb = sv.spec_verify_workspace_bytes(sv.MODE_REJECTION, Bt, kt, Vt)
    ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
    flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def standard():
        check(lib.spec_verify_rejection(P(inp.logits), sv.FP32, P(inp.drafts), P(inp.q), Bt, kt, Vt,
                                        inp.temperature, inp.seed, 3, P(o), P(al), None, P(ws), nb, P(status),
                                        cur()), "spec_verify_rejection")

    def greedy():
        check(lib.spec_verify_greedy(P(inp.logits), sv.FP32, P(inp.drafts), Bt, kt, Vt, P(o), P(al), P(ws), nb,
                                     P(status), cur()), "spec_verify_greedy")

    res = {}
    for name, fn, launches in (("tiny_standard", standard, 3), ("tiny_greedy", greedy, 2)):
        ms = graph_time_ms(torch, [fn], 50, flush=lambda: flush_buf.zero_())
        res[name] = {"ms_per_call": ms, "us_per_call": ms * 1e3, "positions_per_s": Bt * (kt + 1) / (ms * 1e-3),
                     "launches_per_call": launches,
                     "note": "B=4, k=3, V=1024 fp32: latency-bound, reported as latency; L2 flushed before each call"}
    return res


SWEEP_B = (1, 8, 32, 64, 512)
SWEEP_K = (0, 1, 3, 7)
SWEEP_ALPHA = (0.35, 0.7)


def _sweep_modes(torch, sv, wl, dev, lib, P, cur, check, status, peak):
    """The adaptive-schedule grid: B x k x alpha, standard rejection with draft distributions,
    V=128256 bf16, T=1.  Cells whose logits and q together are under 2/3 of L2 are timed one call
    at a time with L2 flushed before each; larger cells rotate three input sets.  Each cell reports
    positions/s, GB/s against the bytes the rule must read (the logits, q at the drafts, and the q
    row of each request whose round stops at a rejection), and beside it the count with all of q."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    res = {}
    for Bs in SWEEP_B:
        for ks in SWEEP_K:
            for a in SWEEP_ALPHA:
                all_q = chain_bytes(Bs, ks, V, 2, with_q=True)
                rotate = all_q * 3 >= 2 * l2
                nsets = N_SETS if rotate else 1
                sets = [wl.chain_sweep(dev, seed=11000 + 97 * i, B=Bs, k=ks, alpha=a) for i in range(nsets)]
                o = torch.empty((Bs, ks + 1), dtype=torch.int32, device=dev)
                al = torch.empty(Bs, dtype=torch.int32, device=dev)
                nb = sv.spec_verify_workspace_bytes(sv.MODE_REJECTION, Bs, ks, V)
                ws = torch.zeros(nb, dtype=torch.uint8, device=dev)

                def call(i, Bs=Bs, ks=ks, sets=sets, o=o, al=al, ws=ws, nb=nb):
                    x = sets[i % len(sets)]
                    check(lib.spec_verify_rejection(P(x.logits), sv.BF16, P(x.drafts), P(x.q) if ks > 0 else None,
                                                    Bs, ks, V, 1.0, x.seed, i, P(o), P(al), None, P(ws), nb,
                                                    P(status), cur()), "spec_verify_rejection")

                if rotate:
                    ms = graph_time_ms(torch, [lambda i=i: call(i) for i in range(12)], 10)
                else:
                    ms = graph_time_ms(torch, [lambda: call(0)], 20, flush=lambda: flush_buf.zero_())
                nrej = 0
                for i, x in enumerate(sets):
                    call(i)
                    torch.cuda.synchronize()
                    nrej += rejected_rows(al, ks, x.drafts) if ks > 0 else 0
                nrej = nrej / len(sets)
                need = required_bytes(Bs, ks, V, 2, nrej)
                gbs = need / (ms * 1e-3) / 1e9
                res[f"sweep_B{Bs}_k{ks}_a{a}"] = {
                    "B": Bs, "k": ks, "alpha": a, "ms_per_call": ms, "positions_per_s": Bs * (ks + 1) / (ms * 1e-3),
                    "bytes_required": need, "gbs": gbs, "frac_of_peak": gbs / peak,
                    "rejected_rows_per_call": nrej, "bytes_all_of_q": all_q,
                    "gbs_all_of_q": all_q / (ms * 1e-3) / 1e9,
                    "l2": "3 rotating input sets" if rotate else "L2 flushed before each call",
                    "launches_per_call": 3 if ks > 0 else 2}
                del sets, ws
    return res


def _variant_modes(torch, sv, wl, dev, lib, P, cur, check, status, out, alen, peak):
    """Verify variants on the headline workload: a temperature per request (every other request
    greedy, the rest sampling at T in [0.6, 1.4]), relaxed thresholds (0.5, 0.5), top-k 50 with
    top-p 0.9 on every request, and top-p 0.9 alone."""
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
            "top_k50_top_p0.9_b64k7": sv.Options(None, 1.0, 1.0, 1.0, top_k.data_ptr(), top_p.data_ptr()),
            "top_p0.9_b64k7": sv.Options(None, 1.0, 1.0, 1.0, None, top_p.data_ptr())}
    for name, opt in opts.items():
        def call(i, opt=opt):
            x = sets[i % N_SETS]
            check(lib.spec_verify_rejection_ex(P(x.logits), sv.BF16, P(x.drafts), None, B, K_DRAFTS, V,
                                               ct.byref(opt), x.seed, i, P(out), P(alen), None, P(ws), nb,
                                               P(status), cur()), "spec_verify_rejection_ex")

        ms = graph_time_ms(torch, [lambda i=i: call(i) for i in range(GRAPH_CALLS)], 20)
        launches = 4 if name.startswith("top_") else 2
        res[name] = _mode_entry(ms, B * (K_DRAFTS + 1), chain_bytes(B, K_DRAFTS, V, 2), peak, launches,
                                note=("thresholds first: the one-read ring kernel, then the general kernel for the "
                                      "rows it leaves (top-p alone: all of them)") if launches == 4 else None)
    return res


def _budget_modes(torch, sv, dev, lib, P, cur, check, shapes=((512, 7), (2048, 8))):
    """The adaptive verification budget (keys, rank, pick) on B x K slots of random confidences
    with a roofline-shaped cost table; latency per plan."""
    res = {}
    g = torch.Generator(device=dev).manual_seed(5)
    for B_, K_ in shapes:
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
                                          "launches_per_call": 1,
                                          "note": "latency-bound: one cluster of 8 CTAs sorts, scans, picks and admits in distributed shared memory"}
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
    # The same inputs as our arm's first input set (drawn on the GPU when there is one, since the
    # generator's stream differs per device).
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = wl.chain_b64k7(gen_dev, seed=1236 + 7919 * D.rank)
    lg = wl.to_numpy_logits(inp.logits)
    d = inp.drafts.cpu().numpy()

    import concurrent.futures as cf

    threads = os.cpu_count() or 1
    pool = cf.ThreadPoolExecutor(max_workers=threads)
    groups = [np.arange(B, dtype=np.int32)[g::threads] for g in range(threads)]
    groups = [g for g in groups if g.size]

    def step(s):
        # One step verifies the whole batch (B requests), the requests split over the host threads
        # (the oracle's C code runs without the GIL).
        list(pool.map(lambda ids: oracle.verify_rejection(lg, d, None, 1.0, inp.seed, s, req_ids=ids), groups))

    for w in range(args.warmup):
        step(w)
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(args.warmup + s)
    el = time.perf_counter() - t0
    pool.shutdown()
    value = B * (K_DRAFTS + 1) * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": D.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "k": K_DRAFTS, "V": V, "logits": "bf16",
                   "mode": "target-only (one-hot q)", "positions_per_step": B * (K_DRAFTS + 1),
                   "step": f"the whole batch of {B} requests per step, split over {len(groups)} host threads"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": len(groups), "kind": "oracle",
                         "sample": f"{args.steps} steps, each the whole b64k7 batch ({B} requests, "
                                   f"{B * (K_DRAFTS + 1)} positions)"},
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
