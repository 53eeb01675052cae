"""Benchmark of the GDN verification hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the hot path over one batch of synthetic input:

  chain16      one GDN layer, 1 sequence, a 16-position chain, 16 q/k heads /
               48 value heads, d_k = d_v = 128, bf16 q/k/v, fp32 state:
               gdn_verify_chain + gdn_commit_accepted
  tree22       the same heads over a 22-node draft tree: gdn_verify_tree + commit
  batched8x16  8 sequences x 16-position chains over 48 layers:
               48 x gdn_verify_chain + one gdn_commit_accepted over the 48 layers
  prefill8192  one 8192-token sequence, chunk 64: gdn_prefill_chunked
  batched8x22  8 sequences x 22-node draft trees over 48 layers:
               48 x gdn_verify_tree + one gdn_commit_accepted over the 48 layers
  (and variants: *_replay, *_index, *_f16; see WORKLOADS)

With no --workload the run prints ONE JSON line: the headline is chain16
(the metric is quoted "at block 16"), and the other workloads the metric and
its measurement plan name -- tree22 ("tree 22"), batched8x16 and
prefill8192 -- are measured in the same run and nested under "workloads",
each with its step time and percentiles, its own roofline and its end-to-end
figure, together with the tree variants (binary16 snapshots, checkpoint and
replay, the batched tree).  A workload committed by a copy also reports the
commit kernel's own time and roofline.  --workload NAME measures that one workload alone (for profiling).

Metric: node-heads/s (B x N x Hv per layer call, summed over the step; for
the prefill, token-heads/s).  No step finds its data in L2 (129 MB): the
batched and prefill steps are preceded by a 256 MiB write that is not timed;
a single-sequence step (less than L2) instead rotates, back to back and
unflushed, over enough independent copies of the workload to exceed twice L2.
The K timed steps are bracketed by CUDA events on the launch stream; further
blocks of back-to-back steps (and of the dominant kernel alone) give the
percentiles and the roofline figure.  Under torchrun every rank runs its own
replica (independent sequences, no collective on the data path): weak scaling.

The end-to-end figure goes through the package's public API (bound calls,
one ctypes call per launch): every step copies its inputs from pinned host
memory to the device and its outputs back; each buffer set's step is
captured once into a CUDA graph and the graphs are replayed back to back,
timed on the host clock around the whole run.

--impl reference times the CPU oracle (plain float64 C++, the reference for
every parity test) on this host's cores, on a bounded sample of the same
workload each step.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

HEADS = synthetic.HEADS
FLUSH_BYTES = 256 << 20
L2_BYTES = 129 * 10**6
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# bars the kernels are held to: fraction of the measured HBM copy bandwidth
# (verify, commit) and of the measured dense bf16 tensor throughput (prefill)
TARGETS = {"hbm": 0.70, "tensor": 0.50}
# blocks of back-to-back launches behind the percentiles and the roofline figure
STAT_BLOCKS = 9
KERNEL_BLOCK = 100

METRIC = "GDN verify node-heads/s per layer at block 16 / tree 22; % of GB300 HBM roofline"
HEADLINE = "chain16"
NESTED = ("tree22", "batched8x16", "prefill8192", "tree22_f16", "tree22_replay", "batched8x22",
          "batched8x22_replay")


def hold_device(torch, host_s_per_step, steps):
    """Queue a spin on the device long enough for the host to enqueue all the
    timed steps behind it, so that the steps then run back to back: without
    it a step shorter than its own Python launch cost would be timed with
    the host's launch latency in it.  The spin precedes the first step's
    start event and is not timed."""
    seconds = min(0.5, 0.002 + 2.0 * host_s_per_step * steps)
    torch.cuda._sleep(int(seconds * 2.2e9))


# ------------------------------------------------------------------ workloads
def verify_bytes(B, N, Hk, Hv, dk, dv, in_bytes=2, tree=False, persist=True, snap_bytes=4):
    """Algorithmic HBM bytes of one verify call: every input read once, the
    initial state read once, every output (o and, when persisted, all N
    snapshots) written once."""
    state_in = B * Hv * dk * dv * 4
    snap = B * N * Hv * dk * dv * snap_bytes if persist else 0
    qk = 2 * B * N * Hk * dk * in_bytes
    v = B * N * Hv * dv * in_bytes
    gates = 2 * B * N * Hv * 4
    o = B * N * Hv * dv * 4
    extra = (B * N * 4 * 2) if tree else 0   # parent in, depth out
    return state_in + snap + qk + v + gates + o + extra


def commit_bytes(B, Hv, dk, dv, n_layers=1, snap_bytes=4):
    """Algorithmic HBM bytes of one copy commit: the accepted snapshot of every
    (layer, sequence, head) read once and the cached state written once."""
    return B * Hv * dk * dv * (snap_bytes + 4) * n_layers


def prefill_bytes(T, Hk, Hv, dk, dv, in_bytes=2):
    return (2 * T * Hk * dk * in_bytes + T * Hv * dv * in_bytes + 2 * T * Hv * 4 +
            T * Hv * dv * 4 + 2 * Hv * dk * dv * 4)


def prefill_flops(T, Hk, Hv, dk, dv, C=64):
    """Algorithmic flops of the chunked (WY/UT) form, one multiply-add = 2:
    per chunk and q/k head K K^T and Q K^T (C x C x d_k each); per chunk and
    value head K H, Q H and K^T D' (C x d_k x d_v each) and T X, P Delta
    (C x C x d_v each).  The inverse (C^3/3) and the elementwise work are left
    out; the bf16 hi/lo splits are not counted."""
    n_chunks = -(-T // C)
    per_khead = 2 * (2 * C * C * dk)
    per_vhead = 3 * (2 * C * dk * dv) + 2 * (2 * C * C * dv)
    return n_chunks * (Hk * per_khead + Hv * per_vhead)


WORKLOADS = {
    "chain16": dict(B=1, N=16, tree=False, layers=1,
                    desc="1 sequence x 16-position chain (last committed token + 15 drafts), "
                         "16 q/k heads, 48 value heads, d_k=d_v=128, bf16 q/k/v, fp32 gates "
                         "and state; verify + commit of a seeded accept length"),
    "tree22": dict(B=1, N=22, tree=True, layers=1,
                   desc="1 sequence x 22-node DDTree (parent uniform over earlier nodes, depth "
                        "<= 16), same heads; verify + commit of a seeded node"),
    "batched8x16": dict(B=8, N=16, tree=False, layers=48,
                        desc="8 sequences x 16-position chains, same heads, 48 GDN layers with "
                             "fresh inputs per layer; 48 verifies + one 48-layer commit"),
    "batched8x22": dict(B=8, N=22, tree=True, layers=48,
                        desc="8 sequences x 22-node DDTrees (the same trees in every layer), "
                             "same heads, 48 GDN layers with fresh inputs per layer; 48 tree "
                             "verifies + one 48-layer commit"),
    "batched8x22_replay": dict(B=8, N=22, tree=True, layers=48, replay=True,
                               desc="batched8x22 committed by checkpoint and replay: 48 tree "
                                    "verifies without snapshots (per-block solve), 48 replays "
                                    "of the accepted nodes' ancestor paths"),
    "chain16_replay": dict(B=1, N=16, tree=False, layers=1, replay=True,
                           desc="chain16 committed by checkpoint and replay: verify without "
                                "snapshots, then the accepted prefix re-run from the cached "
                                "state into the cache"),
    "batched8x16_replay": dict(B=8, N=16, tree=False, layers=48, replay=True,
                               desc="batched8x16 committed by checkpoint and replay: 48 verifies "
                                    "without snapshots, 48 replays of the accepted prefixes"),
    "chain16_index": dict(B=1, N=16, tree=False, layers=1, index=True,
                          desc="chain16 committed through the index table: verify reads its "
                               "state from the previous block's snapshot region and writes "
                               "its own snapshots there; commit sets slot[b] = b*N + accept"),
    "batched8x16_index": dict(B=8, N=16, tree=False, layers=48, index=True,
                              desc="batched8x16 committed through the index table: 48 verifies "
                                   "on per-layer snapshot regions, one slot table for all "
                                   "layers"),
    "chain16_f16": dict(B=1, N=16, tree=False, layers=1, snap16=True,
                        desc="chain16 persisting binary16 snapshots (gdn_verify_chain_f16) "
                             "and committing by widening (gdn_commit_accepted_f16)"),
    "batched8x16_f16": dict(B=8, N=16, tree=False, layers=48, snap16=True,
                            desc="batched8x16 persisting binary16 snapshots, 48-layer "
                                 "widening commit"),
    "tree22_f16": dict(B=1, N=22, tree=True, layers=1, snap16=True,
                       desc="tree22 persisting binary16 snapshots (gdn_verify_tree_f16, the "
                            "per-block solve that never reads a persisted state back) and "
                            "committing by widening (gdn_commit_accepted_f16)"),
    "tree22_replay": dict(B=1, N=22, tree=True, layers=1, replay=True,
                          desc="tree22 committed by checkpoint and replay: the tree verified "
                               "without snapshots, then the accepted node's ancestors re-run "
                               "from the cached state into the cache"),
    "prefill8192": dict(T=8192, layers=1,
                        desc="1 sequence of 8192 tokens, 16 q/k heads, 48 value heads, "
                             "d_k=d_v=128, bf16 q/k/v, chunk 64, WY/UT form on tensor cores"),
}


def stats_ms(values, how):
    """Summary of per-step (or per-launch) times in ms."""
    v = [float(x) for x in values]
    return {"mean": statistics.mean(v), "p10": float(np.percentile(v, 10)),
            "p50": float(np.percentile(v, 50)), "p90": float(np.percentile(v, 90)),
            "samples": len(v), "how": how}


def roofline_entry(bound, kernel, work_per_launch, launch_ms, peak, peak_kind, traffic,
                   work_key):
    """achieved = algorithmic work per launch / launch time, against the
    measured peak, with the bar the kernel is held to."""
    unit = "GB/s" if bound == "hbm" else "TFLOP/s"
    scale = 1e9 if bound == "hbm" else 1e12
    achieved = work_per_launch / (launch_ms / 1e3) / scale
    frac = achieved / peak
    return {"bound": bound, "kernel": kernel, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": frac, "target": TARGETS[bound], "target_met": frac >= TARGETS[bound],
            "peak_source": (f"{peak_kind} (MEASURED_PEAKS.json "
                            f"{'hbm_gbs' if bound == 'hbm' else 'bf16_tflops'})"
                            if peak_kind == "measured" else f"fallback {peak} {unit}"),
            work_key: work_per_launch, "launch_ms": launch_ms, "traffic": traffic,
            "traffic_over_algorithmic": (traffic / work_per_launch
                                         if traffic is not None and bound == "hbm" else None)}


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background; each line is stamped
    on arrival so the samples inside the timed region can be picked out."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.gpu_id is not None:
                cmd += ["-i", str(self.gpu_id)]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for ts, s in self.samples if t0 <= ts <= t1]
        if not inside and self.samples:   # nearest sample to the window
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda x: abs(x[0] - mid))[1]]
        sm, mx, reasons = [], [], set()
        for s in inside:
            try:
                sm.append(float(s[0]))
                mx.append(float(s[1]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(self.NAMES, s[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside)}


# ---------------------------------------------------------------- roofline
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "verify": ["hybrid_gated_deltanet_delta_gb300/csrc/gdn_verify.cu",
               "hybrid_gated_deltanet_delta_gb300/csrc/gdn_common.cuh"],
    "commit": ["hybrid_gated_deltanet_delta_gb300/csrc/gdn_commit.cu",
               "hybrid_gated_deltanet_delta_gb300/csrc/gdn_common.cuh"],
    "prefill": ["hybrid_gated_deltanet_delta_gb300/csrc/gdn_prefill.cu",
                "hybrid_gated_deltanet_delta_gb300/csrc/gdn_common.cuh",
                "hybrid_gated_deltanet_delta_gb300/csrc/gdn_tc.cuh"],
}


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch recorded by an ncu capture in profiles/, if the
    kernel's sources are unchanged since (source hash in the summary)."""
    sha = source_sha(KERNEL_SOURCES[kernel])
    pat = re.compile(r"bench-traffic: kernel=(\S+) workload=(\S+) source_sha=(\S+) "
                     r"dram_bytes_per_launch=(\d+)")
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".md", ".txt")):
            continue
        for m in pat.finditer(open(os.path.join(pdir, name)).read()):
            if m.group(1) == kernel and m.group(2) == workload and m.group(3) == sha:
                return int(m.group(4))
    return None


# ------------------------------------------------------------------ oracle leg
def host_cpu():
    """(logical cores, CPU model) of this host."""
    cores = os.cpu_count() or 1
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu model")):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return cores, model or "unknown"


class OracleSampler:
    """Bounded samples of a workload for the oracle.  A verify sample is value
    heads h .. h+n-1 (wrapping) of sequence 0 of one layer, verified and then
    committed (copy, or replay for the *_replay workloads); a prefill sample
    is one value head over all 8192 tokens in the step form."""

    def __init__(self, wl_name):
        self.wl = wl_name
        self.prefill = wl_name == "prefill8192"
        if self.prefill:
            self.inp = synthetic.prefill8192()
        elif wl_name.startswith("chain16"):
            self.inp = synthetic.chain16()
        elif wl_name.startswith("tree22"):
            self.inp = synthetic.tree22()
        elif wl_name.startswith("batched8x22"):
            self.inp = synthetic.batched8x22_layer(0)
        else:
            self.inp = synthetic.batched8x16_layer(0)

    @property
    def unit(self):
        return "token-heads/s" if self.prefill else "node-heads/s"

    def run(self, h0=0, n_heads=1):
        """One sample; returns the node-heads (token-heads) it covered."""
        import oracle

        inp = self.inp
        if self.prefill:
            h = h0 % inp["Hv"]
            st, _, _ = oracle.prefill_step(inp["q_f64"], inp["k_f64"], inp["v_f64"],
                                           inp["alpha"], inp["beta"], inp["state"], T=inp["T"],
                                           Hk=inp["Hk"], Hv=inp["Hv"], dk=inp["dk"],
                                           dv=inp["dv"], heads=(h, 1))
            assert st == oracle.OK
            return inp["T"]
        b = 0
        N = inp["N"]
        h_sel = (h0 + np.arange(n_heads)) % inp["Hv"]
        G = inp["Hv"] // inp["Hk"]
        hk_sel = h_sel // G
        q = inp["q_f64"][b:b + 1][:, :, hk_sel]
        k = inp["k_f64"][b:b + 1][:, :, hk_sel]
        v = inp["v_f64"][b:b + 1][:, :, h_sel]
        al = inp["alpha"][b:b + 1][:, :, h_sel]
        be = inp["beta"][b:b + 1][:, :, h_sel]
        cache = inp["cache"][inp["slot"][b]][h_sel][None]
        parent = inp["parent"][b:b + 1] if inp["tree"] else None
        st, snap, _ = oracle.verify(q, k, v, al, be, cache, np.zeros(1, np.int32), parent, B=1,
                                    N=N, Hk=n_heads, Hv=n_heads, dk=inp["dk"], dv=inp["dv"])
        assert st == oracle.OK
        if self.wl.endswith("_replay"):
            dst = np.ascontiguousarray(cache, dtype=np.float64).copy()
            st = oracle.replay(k, v, al, be, dst, np.zeros(1, np.int32), parent,
                               inp["accept"][b:b + 1], B=1, N=N, Hk=n_heads, Hv=n_heads,
                               dk=inp["dk"], dv=inp["dv"])
        else:
            dst = np.zeros((1, n_heads, inp["dk"], inp["dv"]))
            st = oracle.commit(snap, inp["accept"][b:b + 1], dst, None, B=1, N=N, Hv=n_heads,
                               dk=inp["dk"], dv=inp["dv"])
        assert st == oracle.OK
        return N * n_heads

    def describe(self, n_heads):
        if self.prefill:
            return "8192 tokens x 1 value head (step form, float64)"
        return (f"verify + commit of {n_heads} value head(s) x {self.inp['N']} nodes of "
                f"sequence 0, float64")

    def timed(self, budget_s, threads, n_heads=3):
        """Samples on `threads` host threads (each its own value heads; the
        oracle's C calls release the interpreter lock) until about budget_s
        seconds have passed; returns (units per second, samples)."""
        done, reps = 0, 0
        t0 = time.perf_counter()
        if threads == 1:
            while time.perf_counter() - t0 < budget_s or reps == 0:
                done += self.run(reps * n_heads, n_heads)
                reps += 1
        else:
            with cf.ThreadPoolExecutor(max_workers=threads) as ex:
                while time.perf_counter() - t0 < budget_s or reps == 0:
                    futs = [ex.submit(self.run, (reps + i) * n_heads, n_heads)
                            for i in range(threads)]
                    done += sum(f.result() for f in futs)
                    reps += threads
        spent = time.perf_counter() - t0
        return done / spent, reps


def cpu_baseline(wl_name, budget_s=8.0):
    """The oracle as it stands on this host: all cores (a thread pool over
    independent value heads, the reported value) and one thread beside it."""
    smp = OracleSampler(wl_name)
    cores, model = host_cpu()
    n_heads = 1 if smp.prefill else 3
    multi, reps_m = smp.timed(budget_s, cores, n_heads)
    single, reps_s = smp.timed(budget_s, 1, n_heads)
    return {"value": multi, "unit": smp.unit, "cores": cores, "kind": "oracle",
            "sample": f"{reps_m} samples on {cores} threads, each {smp.describe(n_heads)}",
            "cpu_model": model, "host_cores": cores,
            "single_thread": {"value": single, "cores": 1,
                              "sample": f"{reps_s} samples, each {smp.describe(n_heads)}"}}


# ----------------------------------------------------------------- ours: GPU
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _dev(a, torch):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class VerifyCase:
    """Device buffers for one verify layer (inputs, cache, outputs).  The
    per-step inputs (q, k, v, alpha, beta, accept) live in one packed device
    buffer so that the end-to-end leg moves them with a single copy from one
    pinned host buffer."""

    NAMES = ("q", "k", "v", "alpha", "beta", "accept")   # and a tree's parent array

    def __init__(self, inp, torch, pinned=False, persist=True, snap16=False):
        self.inp = inp
        self.snap16 = snap16
        self.B, self.N, self.Hv = inp["B"], inp["N"], inp["Hv"]
        dk, dv = inp["dk"], inp["dv"]
        names = self.NAMES + (("parent",) if inp["tree"] else ())
        arrays = {n: np.ascontiguousarray(inp[n]) for n in names}
        offs, total = {}, 0
        for n in names:
            offs[n] = total
            total += (arrays[n].nbytes + 255) // 256 * 256
        host = np.zeros(total, np.uint8)
        for n in names:
            host[offs[n]:offs[n] + arrays[n].nbytes] = arrays[n].view(np.uint8).ravel()
        self.packed = torch.from_numpy(host).cuda()
        tdt = {np.dtype(np.uint16): torch.bfloat16, np.dtype(np.float32): torch.float32,
               np.dtype(np.int32): torch.int32}
        self.dev = {}
        for n in names:
            a = arrays[n]
            seg = self.packed[offs[n]:offs[n] + a.nbytes]
            self.dev[n] = seg.view(tdt[a.dtype]).view(*a.shape)
        self.cache = _dev(inp["cache"], torch)
        self.slot = _dev(inp["slot"], torch)
        self.parent = self.dev["parent"] if inp["tree"] else None
        self.snap = (torch.empty((self.B, self.N, self.Hv, dk, dv), device="cuda",
                                 dtype=torch.float16 if snap16 else torch.float32)
                     if persist else None)
        self.o = torch.empty((self.B, self.N, self.Hv, dv), device="cuda")
        self.host = None
        if pinned:
            self.host = self.packed.cpu().pin_memory()
            self.o_host = torch.empty(self.o.shape, dtype=torch.float32).pin_memory()

    def verify(self, gdn):
        """The binding's plain (checked) call."""
        d = self.dev
        args = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], self.cache, self.snap, self.o)
        if self.snap16 and self.parent is not None:
            gdn.gdn_verify_tree_f16(*args, self.parent, slot=self.slot,
                                    n_slots=self.inp["n_slots"])
        elif self.snap16:
            gdn.gdn_verify_chain_f16(*args, slot=self.slot, n_slots=self.inp["n_slots"])
        elif self.parent is not None:
            gdn.gdn_verify_tree(*args, self.parent, slot=self.slot, n_slots=self.inp["n_slots"])
        else:
            gdn.gdn_verify_chain(*args, slot=self.slot, n_slots=self.inp["n_slots"])

    def replay(self, gdn):
        """The binding's plain (checked) replay commit."""
        d = self.dev
        gdn.gdn_replay_accepted(d["k"], d["v"], d["alpha"], d["beta"], self.cache, d["accept"],
                                parent=self.parent, slot=self.slot,
                                n_slots=self.inp["n_slots"])

    def bind(self, gdn, stream):
        """This layer's verify and replay as bound calls (the package's public
        serving API: arguments marshalled once, one ctypes call per launch)."""
        d = self.dev
        n_slots = self.inp["n_slots"]
        common = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], self.cache)
        if self.snap16 and self.parent is not None:
            self.verify_c = gdn.bind_verify_tree(*common, None, self.o, self.parent,
                                                 snapshots_f16=self.snap, slot=self.slot,
                                                 n_slots=n_slots, stream=stream)
        elif self.snap16:
            self.verify_c = gdn.bind_verify_chain(*common, None, self.o, snapshots_f16=self.snap,
                                                  slot=self.slot, n_slots=n_slots, stream=stream)
        elif self.parent is not None:
            self.verify_c = gdn.bind_verify_tree(*common, self.snap, self.o, self.parent,
                                                 slot=self.slot, n_slots=n_slots, stream=stream)
        else:
            self.verify_c = gdn.bind_verify_chain(*common, self.snap, self.o, slot=self.slot,
                                                  n_slots=n_slots, stream=stream)
        self.replay_c = gdn.bind_replay_accepted(d["k"], d["v"], d["alpha"], d["beta"],
                                                 self.cache, d["accept"], parent=self.parent,
                                                 slot=self.slot, n_slots=n_slots, stream=stream)

    def h2d(self):
        self.packed.copy_(self.host, non_blocking=True)
        return self.host.numel()

    def d2h(self):
        self.o_host.copy_(self.o, non_blocking=True)
        return self.o.numel() * 4


class Context:
    """What every measurement shares: the library, the stream, the L2 flush
    buffer, the clock sampler and the rank layout."""

    def __init__(self, args, world, rank, local):
        import torch

        import hybrid_gated_deltanet_delta_gb300 as gdn

        self.args, self.world, self.rank, self.local = args, world, rank, local
        self.torch, self.gdn = torch, gdn
        torch.cuda.set_device(local)
        gdn.load()
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        self.stream = torch.cuda.current_stream()
        self.flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.sampler = ClockSampler(gpu_uuid(torch, local))
        self.sampler.start()
        self.peaks = measured_peaks()

    def close(self):
        self.sampler.stop()

    def events(self, n):
        return [self.torch.cuda.Event(enable_timing=True) for _ in range(n)]


TREE_WARPS = 4      # warps of a tree verify block
TREE_STASH_SLOTS = 3


def tree_walk_stats(parent):
    """Rounds and parent reads of the level-by-level tree walk for one tree:
    the warps of a block take each depth level's nodes round robin (index
    order); a node finds its parent in its warp's registers (the warp formed
    it last), in the shared-memory stash (the first TREE_STASH_SLOTS nodes
    of a level that have children), or reads it back through L2."""
    N = len(parent)
    depth = [0] * N
    for n in range(N):
        depth[n] = 1 if parent[n] < 0 else depth[parent[n]] + 1
    has_child = [False] * N
    for n in range(1, N):
        has_child[parent[n]] = True
    stashed = [has_child[n] and sum(1 for m in range(n) if has_child[m] and depth[m] == depth[n])
               < TREE_STASH_SLOTS for n in range(N)]
    held = [-1] + [-2] * (TREE_WARPS - 1)
    rounds = l2 = 0
    for d in range(1, max(depth) + 1):
        level = [n for n in range(N) if depth[n] == d]
        rounds += (len(level) + TREE_WARPS - 1) // TREE_WARPS
        for i, n in enumerate(level):
            w = i % TREE_WARPS
            if parent[n] >= 0 and held[w] != parent[n] and not stashed[parent[n]]:
                l2 += 1
            held[w] = n
    return {"depth": max(depth), "rounds": rounds, "parents_read_from_l2": l2}


def tree_shape_sweep(ctx, n_trees=16, copies=4, launches=100):
    """The tree22 verify on other seeded 22-node trees (same generator, same
    head shapes): per-launch time back to back over rotating copies larger
    than L2, with each tree's walk statistics."""
    torch, gdn, stream = ctx.torch, ctx.gdn, ctx.stream
    base = synthetic.workload_seed("tree22")
    rows = []
    for t in range(1, n_trees + 1):
        inp = synthetic.tree22(seed=base + 0x1000 + t)
        cases = [VerifyCase(inp, torch) for _ in range(copies)]
        calls = [gdn.bind_verify_tree(c.dev["q"], c.dev["k"], c.dev["v"], c.dev["alpha"],
                                      c.dev["beta"], c.cache, c.snap, c.o, c.parent,
                                      slot=c.slot, n_slots=inp["n_slots"], stream=stream)
                 for c in cases]
        for i in range(20):
            calls[i % copies]()
        torch.cuda.synchronize()
        hold_device(torch, 20e-6, launches)
        e = ctx.events(2)
        e[0].record(stream)
        for i in range(launches):
            calls[i % copies]()
        e[1].record(stream)
        torch.cuda.synchronize()
        row = tree_walk_stats([int(x) for x in inp["parent"][0]])
        row["verify_us"] = e[0].elapsed_time(e[1]) / launches * 1e3
        rows.append(row)
        del cases, calls
    us = sorted(r["verify_us"] for r in rows)
    return {"trees": n_trees, "verify_us_min": us[0], "verify_us_p50": us[len(us) // 2],
            "verify_us_max": us[-1], "per_tree": rows,
            "how": f"tree22's generator with {n_trees} other seeds; per tree {launches} "
                   f"back-to-back verify launches over {copies} rotating copies, one event "
                   "pair; rounds and parent reads through L2 of the level walk"}


def measure_verify(ctx, wl_name):
    torch, gdn, args, stream, flush = ctx.torch, ctx.gdn, ctx.args, ctx.stream, ctx.flush
    world = ctx.world
    wl = WORKLOADS[wl_name]
    Hk, Hv, dk, dv = HEADS["Hk"], HEADS["Hv"], HEADS["dk"], HEADS["dv"]
    B, N = wl["B"], wl["N"]
    replay = wl.get("replay", False)
    index = wl.get("index", False)
    snap16 = wl.get("snap16", False)
    tree = wl.get("tree", False)
    batched = wl_name.startswith("batched")
    L = args.layers if (args.layers and batched) else wl["layers"]
    vbytes = verify_bytes(B, N, Hk, Hv, dk, dv, tree=tree, persist=not replay,
                          snap_bytes=2 if snap16 else 4)
    if batched:
        # every step moves far more than L2; the flush before it is not timed
        n_sets, flush_each = 1, True
    else:
        # a single-sequence step touches less than L2: the steps rotate over
        # independent copies of the workload, together more than twice L2,
        # back to back with no flush in between
        step_bytes = vbytes + commit_bytes(B, Hv, dk, dv)
        n_sets, flush_each = min(64, max(2, -(-2 * L2_BYTES // step_bytes))), False

    def make_set():
        """Buffers of one copy of the workload and its step (verify, commit)."""
        ws = argparse.Namespace()
        if batched:
            layer_inputs = synthetic.batched8x22_layer if tree else synthetic.batched8x16_layer
            ws.layers = [VerifyCase(layer_inputs(l), torch, pinned=True,
                                    persist=not replay, snap16=snap16) for l in range(L)]
            # one cache for all layers: [layer][slot][Hv][dk][dv]; snapshots likewise
            ws.cache_all = torch.stack([c.cache for c in ws.layers])
            ws.snap_all = None if replay else torch.empty(
                (L, B, N, Hv, dk, dv), device="cuda",
                dtype=torch.float16 if snap16 else torch.float32)
            for l, c in enumerate(ws.layers):
                c.cache = ws.cache_all[l]
                if not replay:
                    c.snap = ws.snap_all[l]
        else:
            inp = synthetic.tree22() if tree else synthetic.chain16()
            ws.layers = [VerifyCase(inp, torch, pinned=True, persist=not replay, snap16=snap16)]
            ws.cache_all = ws.layers[0].cache
            ws.snap_all = ws.layers[0].snap
        ws.accept = ws.layers[0].dev["accept"]
        ws.slot = ws.layers[0].slot
        if index:
            # the first verify of every layer reads the cache; afterwards each
            # layer's snapshot region is its cache, addressed through one slot table
            for c in ws.layers:
                c.verify(gdn)
            ws.slot_idx = torch.empty(B, dtype=torch.int32, device="cuda")
            gdn.gdn_commit_index(ws.accept, ws.slot_idx, N=N)
            for c in ws.layers:
                c.cache = c.snap.view(B * N, Hv, dk, dv)
                c.slot = ws.slot_idx
                c.inp = dict(c.inp, n_slots=B * N)
            torch.cuda.synchronize()
        ws.cache_init = None if index else ws.cache_all.clone()
        return ws

    def commit(ws):
        """The binding's plain (checked) commit of a set."""
        if index:
            gdn.gdn_commit_index(ws.accept, ws.slot_idx, N=N)
        elif replay:
            for c in ws.layers:
                c.replay(gdn)
        else:
            gdn.gdn_commit_accepted(ws.snap_all, ws.accept, ws.cache_all, B=B, N=N, Hv=Hv, dk=dk,
                                    dv=dv, n_layers=len(ws.layers),
                                    snap_layer_stride=B * N * Hv * dk * dv,
                                    cache_layer_stride=B * Hv * dk * dv, slot=ws.slot, n_slots=B)

    def bind_set(ws):
        """The set's step as bound calls."""
        for c in ws.layers:
            c.bind(gdn, stream)
        if index:
            ws.commit_c = [lambda: gdn.gdn_commit_index(ws.accept, ws.slot_idx, N=N,
                                                        stream=stream)]
        elif replay:
            ws.commit_c = [c.replay_c for c in ws.layers]
        else:
            ws.commit_c = [gdn.bind_commit_accepted(
                ws.snap_all, ws.accept, ws.cache_all, B=B, N=N, Hv=Hv, dk=dk, dv=dv,
                n_layers=len(ws.layers), snap_layer_stride=B * N * Hv * dk * dv,
                cache_layer_stride=B * Hv * dk * dv, slot=ws.slot, n_slots=B, stream=stream)]
        ws.verify_c = [c.verify_c for c in ws.layers]

    def bind_calls(ws, on_stream):
        """The set's step (verifies, then commit) as bound calls on another stream."""
        out = []
        for c in ws.layers:
            d = c.dev
            common = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], c.cache)
            kw = dict(slot=c.slot, n_slots=c.inp["n_slots"], stream=on_stream)
            if c.snap16 and c.parent is not None:
                out.append(gdn.bind_verify_tree(*common, None, c.o, c.parent,
                                                snapshots_f16=c.snap, **kw))
            elif c.snap16:
                out.append(gdn.bind_verify_chain(*common, None, c.o, snapshots_f16=c.snap, **kw))
            elif c.parent is not None:
                out.append(gdn.bind_verify_tree(*common, c.snap, c.o, c.parent, **kw))
            else:
                out.append(gdn.bind_verify_chain(*common, c.snap, c.o, **kw))
        if index:
            out.append(lambda: gdn.gdn_commit_index(ws.accept, ws.slot_idx, N=N,
                                                    stream=on_stream))
        elif replay:
            for c in ws.layers:
                d = c.dev
                out.append(gdn.bind_replay_accepted(d["k"], d["v"], d["alpha"], d["beta"],
                                                    c.cache, d["accept"], parent=c.parent,
                                                    slot=c.slot, n_slots=c.inp["n_slots"],
                                                    stream=on_stream))
        else:
            out.append(gdn.bind_commit_accepted(
                ws.snap_all, ws.accept, ws.cache_all, B=B, N=N, Hv=Hv, dk=dk, dv=dv,
                n_layers=len(ws.layers), snap_layer_stride=B * N * Hv * dk * dv,
                cache_layer_stride=B * Hv * dk * dv, slot=ws.slot, n_slots=B, stream=on_stream))
        return out

    def step_c(ws, ev=None):
        """One step through the bound calls; ev = (start, after verify, end)."""
        if ev is not None:
            ev[0].record(stream)
        for f in ws.verify_c:
            f()
        if ev is not None:
            ev[1].record(stream)
        for f in ws.commit_c:
            f()
        if ev is not None:
            ev[2].record(stream)

    sets = [make_set() for _ in range(n_sets)]
    for ws in sets:
        bind_set(ws)
    layers = sets[0].layers
    launches_per_step = len(layers) * 2 if replay else len(layers) + 1
    # warm-up: the binding's checked calls once per set, then the bound calls
    for ws in sets:
        for c in ws.layers:
            c.verify(gdn)
        commit(ws)
    n_warm = max(args.warmup, n_sets)
    th = time.perf_counter()
    for i in range(n_warm):
        if flush_each:
            flush.fill_(1.0)
        step_c(sets[i % n_sets])
    host_s = (time.perf_counter() - th) / n_warm
    torch.cuda.synchronize()

    barrier(world)
    if not flush_each:
        flush.fill_(0.0)  # the first timed step starts from an L2 without its data
    torch.cuda.synchronize()
    t0 = time.time()
    K = args.steps
    if flush_each:
        # the timed K steps, one event pair per step phase; the flush between
        # steps is excluded
        hold_device(torch, host_s, K)
        evs = [ctx.events(3) for _ in range(K)]
        for i in range(K):
            flush.fill_(float(i))
            step_c(sets[i % n_sets], evs[i])
        torch.cuda.synchronize()
        step_list = [e[0].elapsed_time(e[2]) for e in evs]
        kernel_list = [e[0].elapsed_time(e[1]) / len(layers) for e in evs]
        commit_stats = stats_ms([e[1].elapsed_time(e[2]) for e in evs],
                                "commit phase of each timed step")
        total_ms = sum(step_list)
        step_stats = stats_ms(step_list, "one event pair per step (flush before each step "
                                         "not timed)")
        kernel_stats = stats_ms(kernel_list, "verify phase of each timed step / layers")
    else:
        # the timed K steps back to back between one event pair, as a serving
        # loop issues them
        hold_device(torch, host_s, K)
        e_run = ctx.events(2)
        e_run[0].record(stream)
        for i in range(K):
            step_c(sets[i % n_sets])
        e_run[1].record(stream)
        torch.cuda.synchronize()
        total_ms = e_run[0].elapsed_time(e_run[1])
        # percentiles: further blocks of back-to-back steps, one event pair per
        # block (an event between two steps would break the programmatic
        # overlap, so per-step pairs are not used here)
        kb = max(20, K)
        per_step = []
        for r in range(STAT_BLOCKS):
            hold_device(torch, host_s, kb)
            e = ctx.events(2)
            e[0].record(stream)
            for i in range(kb):
                step_c(sets[(r * kb + i) % n_sets])
            e[1].record(stream)
            torch.cuda.synchronize()
            per_step.append(e[0].elapsed_time(e[1]) / kb)
        step_stats = stats_ms(per_step, f"{STAT_BLOCKS} blocks of {kb} back-to-back steps, "
                                        "one event pair per block; per-step mean of each block")
        # the dominant kernel on its own: verify launches back to back over
        # the same rotating copies (every launch again misses L2)
        per_launch = []
        for r in range(STAT_BLOCKS):
            hold_device(torch, host_s / 2, KERNEL_BLOCK)
            e = ctx.events(2)
            e[0].record(stream)
            for i in range(KERNEL_BLOCK):
                for f in sets[(r * KERNEL_BLOCK + i) % n_sets].verify_c:
                    f()
            e[1].record(stream)
            torch.cuda.synchronize()
            per_launch.append(e[0].elapsed_time(e[1]) / (KERNEL_BLOCK * len(layers)))
        kernel_stats = stats_ms(per_launch, f"{STAT_BLOCKS} blocks of {KERNEL_BLOCK} "
                                            "back-to-back verify launches over the rotating "
                                            "copies, one event pair per block")
        # the commit on its own, likewise
        per_commit = []
        for r in range(STAT_BLOCKS):
            hold_device(torch, host_s / 2, KERNEL_BLOCK)
            e = ctx.events(2)
            e[0].record(stream)
            for i in range(KERNEL_BLOCK):
                for f in sets[(r * KERNEL_BLOCK + i) % n_sets].commit_c:
                    f()
            e[1].record(stream)
            torch.cuda.synchronize()
            per_commit.append(e[0].elapsed_time(e[1]) / KERNEL_BLOCK)
        commit_stats = stats_ms(per_commit, f"{STAT_BLOCKS} blocks of {KERNEL_BLOCK} "
                                            "back-to-back commit calls over the rotating "
                                            "copies, one event pair per block")
    barrier(world)
    t1 = time.time()
    total_ms = max_over_ranks(total_ms, world)

    # end to end through the package's calls: every step copies its inputs
    # from pinned host memory, runs the bound verify and commit calls and
    # copies its outputs back.  Each set's step (copies and launches) is
    # captured once into a CUDA graph, as a serving loop would, and the
    # graphs are replayed back to back; host clock around the run.
    for ws in sets:
        if ws.cache_init is not None:
            ws.cache_all.copy_(ws.cache_init)
    e2e_steps = max(K, 50 if batched else 400)
    cap_stream, side = torch.cuda.Stream(), torch.cuda.Stream()
    graphs = []
    h2d = sum(c.host.numel() for c in sets[0].layers)
    d2h = sum(c.o.numel() * 4 for c in sets[0].layers)
    pipelined = n_sets >= 2
    for j, ws in enumerate(sets):
        calls = bind_calls(ws, cap_stream)
        g = torch.cuda.CUDAGraph()
        cap_stream.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap_stream, capture_error_mode="thread_local"):
            if pipelined:
                # this step's launches, and beside them the previous step's
                # outputs out and the next step's inputs in
                side.wait_stream(cap_stream)
                with torch.cuda.stream(side):
                    for c in sets[(j - 1) % n_sets].layers:
                        c.d2h()
                    for c in sets[(j + 1) % n_sets].layers:
                        c.h2d()
                for f in calls:
                    f()
                cap_stream.wait_stream(side)
            else:
                for c in ws.layers:
                    c.h2d()
                for f in calls:
                    f()
                for c in ws.layers:
                    c.d2h()
        graphs.append(g)
    torch.cuda.synchronize()
    for i in range(3):   # warm the graphs
        graphs[i % n_sets].replay()
    torch.cuda.synchronize()
    barrier(world)
    ta = time.perf_counter()
    if pipelined:
        for c in sets[0].layers:   # the first step's inputs
            c.h2d()
    for i in range(e2e_steps):
        graphs[i % n_sets].replay()
    if pipelined:
        for c in sets[(e2e_steps - 1) % n_sets].layers:   # the last step's outputs
            c.d2h()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - ta, world)
    del graphs

    node_heads = B * N * Hv * len(layers)
    hbm, _, peak_kind = ctx.peaks
    kname = ("gdn_verify_tree" if tree else "gdn_verify_chain") + \
        (" (no snapshots)" if replay else " (binary16 snapshots)" if snap16 else
         " (state and snapshots in the slot region)" if index else "") + \
        (", per-block solve" if tree and (replay or snap16) else "")
    out = {
        "metric": METRIC,
        "value": job_throughput(node_heads, K, total_ms, world),
        "unit": "node-heads/s",
        "steps": K,
        "ms_per_step": total_ms / K,
        "step_ms": step_stats,
        "config": {
            "workload": f"{wl_name}: {wl['desc']}",
            "B": B, "N": N, "Hk": Hk, "Hv": Hv, "dk": dk, "dv": dv, "layers": len(layers),
            "inputs": "bf16 q/k/v (L2-normalised q/k), fp32 alpha/beta/state/outputs",
            "node_heads_per_step": node_heads,
            "l2": ("flushed by a 256 MiB write before every step; flush not timed"
                   if flush_each else
                   f"inputs larger than L2: the steps rotate, back to back and unflushed, over "
                   f"{n_sets} independent copies of the workload ({n_sets} x "
                   f"{(vbytes + commit_bytes(B, Hv, dk, dv)) / 1e6:.1f} MB > 2 x 129 MB)"),
            "timing": ("CUDA events on the launch stream around each step's verify and "
                       "commit phases" if flush_each else
                       "CUDA events on the launch stream around the K back-to-back steps"),
            "launch": "programmatic dependent launch (each kernel waits on its predecessor "
                      "before any global-memory access); bound calls, one ctypes call per "
                      "launch",
            "parallelism": f"replicas x{world}, no collective",
        },
        "kernel_ms": kernel_stats,
        "roofline": roofline_entry("hbm", kname, vbytes, kernel_stats["p50"], hbm, peak_kind,
                                   profiled_traffic("verify", wl_name),
                                   "algorithmic_bytes_per_launch"),
        "e2e": {"value": world * node_heads * e2e_steps / e2e_s, "unit": "node-heads/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "how": "per step the packed inputs copied from pinned host memory, the bound "
                       "verify and commit calls, and the outputs o copied back; captured once "
                       "per set into a CUDA graph (with several sets, a step's graph copies the "
                       "previous step's outputs out and the next step's inputs in beside its "
                       "own launches) and replayed back to back; host clock around the run"},
        "gpu_launches": launches_per_step * K,
        "clocks": ctx.sampler.summary(t0, t1),
    }
    if wl_name == "tree22" and world == 1:
        out["shape_sweep"] = tree_shape_sweep(ctx)
    if not (index or replay):
        # the copy commit's own kernel (replay and index commits are other work)
        cbytes = commit_bytes(B, Hv, dk, dv, len(layers), snap_bytes=2 if snap16 else 4)
        out["commit"] = {
            "kernel_ms": commit_stats,
            "roofline": roofline_entry("hbm", "gdn_commit_accepted" + ("_f16" if snap16 else ""),
                                       cbytes, commit_stats["p50"], hbm, peak_kind,
                                       profiled_traffic("commit", wl_name),
                                       "algorithmic_bytes_per_launch")}
    del sets
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def measure_prefill(ctx, wl_name="prefill8192"):
    torch, gdn, args, stream, flush = ctx.torch, ctx.gdn, ctx.args, ctx.stream, ctx.flush
    world = ctx.world
    inp = synthetic.prefill8192()
    T, Hk, Hv, dk, dv = inp["T"], inp["Hk"], inp["Hv"], inp["dk"], inp["dv"]
    q, k, v = (_dev(inp[n], torch) for n in ("q", "k", "v"))
    alpha, beta = _dev(inp["alpha"], torch), _dev(inp["beta"], torch)
    state0 = _dev(inp["state"], torch)
    state = state0.clone()
    o = torch.empty((T, Hv, dv), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wbytes = gdn.gdn_prefill_workspace_bytes(T, Hk, Hv, dk, dv, 64)
    ws = torch.empty(max(wbytes, 16), dtype=torch.uint8, device="cuda")
    call = gdn.bind_prefill_chunked(q, k, v, alpha, beta, state, o, ws, status=status,
                                    stream=stream)

    def step(ev=None):
        state.copy_(state0)
        if ev is not None:
            ev[0].record(stream)
        call()
        if ev is not None:
            ev[1].record(stream)

    gdn.gdn_prefill_chunked(q, k, v, alpha, beta, state, o, ws)   # the checked call once
    th = time.perf_counter()
    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    host_s = (time.perf_counter() - th) / max(1, args.warmup)
    torch.cuda.synchronize()
    K = args.steps
    # the K timed calls, then more for the percentiles, each with its own
    # event pair and the flush before it untimed
    n_stat = max(K, 30)
    evs = [ctx.events(2) for _ in range(K + n_stat)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    hold_device(torch, host_s, K + n_stat)
    for i in range(K + n_stat):
        flush.fill_(float(i))
        step(evs[i])
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    if int(status.item()) != 0:
        raise RuntimeError(f"prefill status {gdn.status_string(int(status.item()))}")
    ms = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = max_over_ranks(sum(ms[:K]), world)
    call_stats = stats_ms(ms, "one event pair per call (prep + scan kernels), 256 MiB flush "
                              "before each call not timed")
    # end to end: host inputs (pinned) -> device -> prefill -> host o and state
    # for every step, each buffer set's step captured once into a CUDA graph
    # and the graphs (two sets) replayed back to back; host clock around the
    # run
    hq, hk, hv, ha, hb = (x.cpu().pin_memory() for x in (q, k, v, alpha, beta))
    hs0 = state0.cpu().pin_memory()
    ho = torch.empty(o.shape).pin_memory()
    hst = torch.empty(state.shape).pin_memory()
    bufs = []
    for j in range(2):
        if j == 0:
            dq, dk_, dv_, da, db, ds, do_, dws, dstat = q, k, v, alpha, beta, state, o, ws, status
        else:
            dq, dk_, dv_, da, db = (torch.empty_like(x) for x in (q, k, v, alpha, beta))
            ds, do_ = torch.empty_like(state), torch.empty_like(o)
            dws, dstat = torch.empty_like(ws), torch.zeros_like(status)
        bufs.append(dict(
            pairs=((dq, hq), (dk_, hk), (dv_, hv), (da, ha), (db, hb), (ds, hs0)), o=do_, state=ds,
            ws=dws, status=dstat))
    pairs = bufs[0]["pairs"]

    cap_stream, side = torch.cuda.Stream(), torch.cuda.Stream()

    def h2d_set(bset):
        for d, h in bset["pairs"]:
            d.copy_(h, non_blocking=True)

    def d2h_set(bset):
        ho.copy_(bset["o"], non_blocking=True)
        hst.copy_(bset["state"], non_blocking=True)

    for j, bset in enumerate(bufs):
        # this step's prefill, and beside it the other set's outputs out and
        # next inputs in
        dq, dk_, dv_, da, db, ds = (d for d, _ in bset["pairs"])
        call_cap = gdn.bind_prefill_chunked(dq, dk_, dv_, da, db, ds, bset["o"], bset["ws"],
                                            status=bset["status"], stream=cap_stream)
        other = bufs[1 - j]
        g = torch.cuda.CUDAGraph()
        cap_stream.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap_stream, capture_error_mode="thread_local"):
            side.wait_stream(cap_stream)
            with torch.cuda.stream(side):
                d2h_set(other)
                h2d_set(other)
            call_cap()
            cap_stream.wait_stream(side)
        bset["graph"] = g
    torch.cuda.synchronize()
    e2e_steps = max(min(K, 40), 10)
    for i in range(2):
        bufs[i]["graph"].replay()
    torch.cuda.synchronize()
    barrier(world)
    ta = time.perf_counter()
    h2d_set(bufs[0])   # the first step's inputs
    for i in range(e2e_steps):
        bufs[i % 2]["graph"].replay()
    d2h_set(bufs[(e2e_steps - 1) % 2])   # the last step's outputs
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - ta, world)
    h2d = sum(h.numel() * h.element_size() for _, h in pairs)
    d2h = ho.numel() * 4 + hst.numel() * 4
    hbm, bf16, kind = ctx.peaks
    pbytes = prefill_bytes(T, Hk, Hv, dk, dv)
    flops = prefill_flops(T, Hk, Hv, dk, dv)
    launch_ms = call_stats["p50"]
    gbs = pbytes / (launch_ms / 1e3) / 1e9
    ptraffic = profiled_traffic("prefill", wl_name)
    out = {
        "metric": METRIC,
        "value": world * T * Hv * K / (total_ms / 1e3),
        "unit": "token-heads/s",
        "steps": K,
        "ms_per_step": total_ms / K,
        "step_ms": call_stats,
        "config": {"workload": f"{wl_name}: {WORKLOADS[wl_name]['desc']}",
                   "T": T, "Hk": Hk, "Hv": Hv, "dk": dk, "dv": dv, "chunk": 64,
                   "l2": "flushed by a 256 MiB write before every call; flush not timed",
                   "timing": "CUDA events around each prefill call (prep + scan kernels) "
                             "on the launch stream",
                   "hbm_achieved_gbs": gbs, "hbm_frac_of_measured": gbs / hbm,
                   "algorithmic_bytes_per_call": pbytes,
                   "dram_traffic_over_algorithmic_bytes": (ptraffic / pbytes
                                                           if ptraffic is not None else None),
                   "workspace_bytes": wbytes},
        "kernel_ms": call_stats,
        "roofline": roofline_entry("tensor", "gdn_prefill_chunked (prep + scan)", flops,
                                   launch_ms, bf16, kind, ptraffic,
                                   "algorithmic_flops_per_launch"),
        "e2e": {"value": world * T * Hv * e2e_steps / e2e_s, "unit": "token-heads/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "how": "per step q, k, v, gates and the initial state copied from pinned host "
                       "memory, the bound prefill call, o and the final state copied back; "
                       "two buffer sets, each step's graph copying the other set's outputs out "
                       "and next inputs in beside its own prefill; graphs replayed back to "
                       "back; host clock around the run"},
        "gpu_launches": 2 * K,   # prep + scan per call
        "clocks": ctx.sampler.summary(t0, t1),
    }
    del ws, o, q, k, v, bufs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def measure(ctx, wl_name):
    if wl_name == "prefill8192":
        return measure_prefill(ctx, wl_name)
    return measure_verify(ctx, wl_name)


def run_ours(args, world, rank, local):
    ctx = Context(args, world, rank, local)
    try:
        name = args.workload or HEADLINE
        out = measure(ctx, name)
        if args.workload is None and not args.no_nested:
            out["workloads"] = {n: measure(ctx, n) for n in NESTED}
    finally:
        ctx.close()
    if rank != 0:
        return None
    line = {"metric": METRIC, "value": out["value"], "unit": out["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": out["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic"}
    line.update({k: v for k, v in out.items() if k not in line})
    return line


def gpu_uuid(torch, local):
    try:
        u = torch.cuda.get_device_properties(local).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:  # noqa: BLE001
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[local]
        return local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The slowest rank's time (host-side control message, not data path)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step_per_rank, steps, max_rank_ms, world):
    """Whole-job units/s: every rank processed the same units; the job took
    as long as its slowest rank."""
    return world * units_per_step_per_rank * steps / (max_rank_ms / 1e3)


# -------------------------------------------------------------- reference arm
def run_reference(args, wl_name, world, rank):
    """The oracle as it stands on this host's cores, each step one bounded
    sample of the workload per host thread."""
    if rank != 0:
        return None
    smp = OracleSampler(wl_name)
    cores, model = host_cpu()
    n_heads = 1 if smp.prefill else 3   # as the cpu_baseline leg samples
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        def one_step(i):
            return sum(f.result() for f in [ex.submit(smp.run, (i * cores + j) * n_heads, n_heads)
                                            for j in range(cores)])
        for i in range(args.warmup):
            one_step(i)
        done = 0
        t0 = time.perf_counter()
        for i in range(args.steps):
            done += one_step(args.warmup + i)
        spent = time.perf_counter() - t0
    value = done / spent
    unit = smp.unit
    sample = f"{cores} samples per step on {cores} threads, each {smp.describe(n_heads)}"
    wl = WORKLOADS[wl_name]
    return {
        "metric": METRIC, "value": value, "unit": unit, "impl": "reference",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * spent / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl_name}: {wl['desc']}"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu_model": model},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=None, choices=sorted(WORKLOADS),
                    help="measure this workload alone (default: chain16 headline with the "
                         "other workloads nested)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0,
                    help="batched8x16 only: run this many of the 48 layers (profiling slices)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (for quick runs)")
    ap.add_argument("--no-nested", action="store_true",
                    help="headline workload only, without the nested workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        out = run_reference(args, args.workload or HEADLINE, world, rank)
    else:
        out = run_ours(args, world, rank, local)
        if out is not None and world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(args.workload or HEADLINE)
            for name, sub in out.get("workloads", {}).items():
                sub["cpu_baseline"] = cpu_baseline(name, budget_s=3.0)
        elif out is not None:
            out["cpu_baseline"] = None
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
