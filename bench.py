"""Benchmark of the GDN verification hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the hot path over one batch of synthetic input:

  chain16      (default) one GDN layer, 1 sequence, a 16-position chain,
               16 q/k heads / 48 value heads, d_k = d_v = 128, bf16 q/k/v,
               fp32 state: gdn_verify_chain + gdn_commit_accepted
  tree22       the same heads over a 22-node draft tree: gdn_verify_tree + commit
  batched8x16  8 sequences x 16-position chains over 48 layers:
               48 x gdn_verify_chain + one gdn_commit_accepted over the 48 layers
  prefill8192  one 8192-token sequence, chunk 64: gdn_prefill_chunked

Metric: node-heads/s (B x N x Hv per layer call, summed over the step; for the
prefill, token-heads/s).  No step finds its data in L2 (129 MB): the batched
and prefill steps are preceded by a 256 MiB write that is not timed; a
single-sequence step (less than L2) instead rotates, back to back and
unflushed, over enough independent copies of the workload to exceed twice L2.
Each step's kernels are bracketed by CUDA events on the launch stream, and the
dominant kernel (the verify / the prefill) by its own pair, which gives the
roofline figure.  Prints ONE JSON
line on rank 0.  Under torchrun every rank runs its own replica (independent
sequences, no collective on the data path): weak scaling.

--impl reference times the CPU oracle (plain float64 C++, the reference for
every parity test) on this host's cores, on a bounded sample of the same
workload each step.
"""
from __future__ import annotations

import argparse
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


def hold_device(torch, host_s_per_step, steps):
    """Queue a spin on the device long enough for the host to enqueue all the
    timed steps behind it, so that the steps then run back to back: without
    it a step shorter than its own Python launch cost would be timed with
    the host's launch latency in it.  The spin precedes the first step's
    start event and is not timed."""
    seconds = min(0.5, 0.002 + 2.0 * host_s_per_step * steps)
    torch.cuda._sleep(int(seconds * 2.2e9))
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

METRIC = "GDN verify node-heads/s per layer at block 16 / tree 22; % of GB300 HBM roofline"


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


def commit_bytes(B, Hv, dk, dv, n_layers=1):
    return 2 * B * Hv * dk * dv * 4 * n_layers


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
    "prefill8192": dict(T=8192, layers=1,
                        desc="1 sequence of 8192 tokens, 16 q/k heads, 48 value heads, "
                             "d_k=d_v=128, bf16 q/k/v, chunk 64, WY/UT form on tensor cores"),
}


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
def oracle_step_sample(wl_name, heads_per_step):
    """The oracle (CPU, float64) on `heads_per_step` value heads of the
    workload's first sequence (one layer), plus the commit of that head:
    returns (seconds, node-heads done)."""
    import oracle

    if wl_name == "prefill8192":
        inp = synthetic.prefill8192()
        t0 = time.perf_counter()
        st, _, _ = oracle.prefill_step(inp["q_f64"], inp["k_f64"], inp["v_f64"], inp["alpha"],
                                       inp["beta"], inp["state"], T=inp["T"], Hk=16, Hv=48,
                                       dk=128, dv=128, heads=(0, heads_per_step))
        assert st == oracle.OK
        return time.perf_counter() - t0, inp["T"] * heads_per_step
    raise NotImplementedError


class OracleSampler:
    """Bounded samples of a verify workload for the oracle: value heads
    h0..h0+G-1 of one q/k head group of sequence 0 (contiguous arrays)."""

    def __init__(self, wl_name):
        self.wl = wl_name
        if wl_name.startswith("chain16"):
            inp = synthetic.chain16()
        elif wl_name == "tree22":
            inp = synthetic.tree22()
        elif wl_name.startswith("batched8x16"):
            inp = synthetic.batched8x16_layer(0)
        else:
            inp = None
        self.inp = inp

    def run(self, n_heads=1):
        """Verify + commit (copy, or replay for the *_replay workloads) for n_heads
        value heads of sequence 0; returns node-heads."""
        import oracle

        inp = self.inp
        b = 0
        N = inp["N"]
        h_sel = np.arange(n_heads) % inp["Hv"]
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


def cpu_baseline(wl_name, budget_s=10.0):
    """The oracle as it stands, single-threaded, repeated on samples of the
    workload until about budget_s seconds of CPU work are done."""
    if wl_name == "prefill8192":
        done, spent, reps = 0, 0.0, 0
        while spent < budget_s or reps == 0:
            dt, n = oracle_step_sample(wl_name, 1)
            spent += dt
            done += n
            reps += 1
        return {"value": done / spent, "unit": "token-heads/s", "cores": 1, "kind": "oracle",
                "sample": f"{reps} x (8192 tokens x 1 value head, step form, float64)"}
    smp = OracleSampler(wl_name)
    heads = 3
    done, reps = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s or reps == 0:
        done += smp.run(heads)
        reps += 1
    spent = time.perf_counter() - t0
    return {"value": done / spent, "unit": "node-heads/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} x (verify + commit of {heads} value heads x {smp.inp['N']} "
                      f"nodes of sequence 0, float64)"}


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

    NAMES = ("q", "k", "v", "alpha", "beta", "accept")

    def __init__(self, inp, torch, pinned=False, persist=True, snap16=False):
        self.inp = inp
        self.snap16 = snap16
        self.B, self.N, self.Hv = inp["B"], inp["N"], inp["Hv"]
        dk, dv = inp["dk"], inp["dv"]
        arrays = {n: np.ascontiguousarray(inp[n]) for n in self.NAMES}
        offs, total = {}, 0
        for n in self.NAMES:
            offs[n] = total
            total += (arrays[n].nbytes + 255) // 256 * 256
        host = np.zeros(total, np.uint8)
        for n in self.NAMES:
            host[offs[n]:offs[n] + arrays[n].nbytes] = arrays[n].view(np.uint8).ravel()
        self.packed = torch.from_numpy(host).cuda()
        tdt = {np.dtype(np.uint16): torch.bfloat16, np.dtype(np.float32): torch.float32,
               np.dtype(np.int32): torch.int32}
        self.dev = {}
        for n in self.NAMES:
            a = arrays[n]
            seg = self.packed[offs[n]:offs[n] + a.nbytes]
            self.dev[n] = seg.view(tdt[a.dtype]).view(*a.shape)
        self.cache = _dev(inp["cache"], torch)
        self.slot = _dev(inp["slot"], torch)
        self.parent = _dev(inp["parent"], torch) if inp["tree"] else None
        self.snap = (torch.empty((self.B, self.N, self.Hv, dk, dv), device="cuda",
                                 dtype=torch.float16 if snap16 else torch.float32)
                     if persist else None)
        self.o = torch.empty((self.B, self.N, self.Hv, dv), device="cuda")
        self.host = None
        if pinned:
            self.host = self.packed.cpu().pin_memory()
            self.o_host = torch.empty(self.o.shape, dtype=torch.float32).pin_memory()

    def verify(self, gdn):
        d = self.dev
        args = (d["q"], d["k"], d["v"], d["alpha"], d["beta"], self.cache, self.snap, self.o)
        if self.snap16:
            gdn.gdn_verify_chain_f16(*args, slot=self.slot, n_slots=self.inp["n_slots"])
        elif self.parent is not None:
            gdn.gdn_verify_tree(*args, self.parent, slot=self.slot, n_slots=self.inp["n_slots"])
        else:
            gdn.gdn_verify_chain(*args, slot=self.slot, n_slots=self.inp["n_slots"])

    def replay(self, gdn):
        d = self.dev
        gdn.gdn_replay_accepted(d["k"], d["v"], d["alpha"], d["beta"], self.cache, d["accept"],
                                parent=self.parent, slot=self.slot,
                                n_slots=self.inp["n_slots"])

    def bind(self, gdn, stream):
        """Marshal this layer's verify and replay once for the timed loop: the
        same C-ABI entry points the binding's functions call, with the
        argument struct built up front, so that a launch costs one ctypes call
        instead of the binding's per-call checks (which would otherwise leave
        the device waiting on the host between short steps)."""
        import ctypes

        lib = gdn.load()
        d = self.dev
        s = ctypes.c_void_p(stream.cuda_stream)

        def ptr(t):
            return None if t is None else ctypes.c_void_p(t.data_ptr())

        n_slots = self.inp["n_slots"]
        self._va = gdn.make_verify_args(d["q"], d["k"], d["v"], d["alpha"], d["beta"], self.cache,
                                        None if self.snap16 else self.snap, self.o,
                                        slot=self.slot, n_slots=n_slots)
        va = ctypes.byref(self._va)
        if self.snap16:
            snap = ptr(self.snap)
            self.verify_c = lambda: lib.gdn_verify_chain_f16(va, snap, s)
        elif self.parent is not None:
            par = ptr(self.parent)
            self.verify_c = lambda: lib.gdn_verify_tree(va, par, None, s)
        else:
            self.verify_c = lambda: lib.gdn_verify_chain(va, s)
        self._ra = gdn.make_verify_args(None, d["k"], d["v"], d["alpha"], d["beta"], self.cache,
                                        None, None, slot=self.slot, n_slots=n_slots)
        ra, par, acc = ctypes.byref(self._ra), ptr(self.parent), ptr(d["accept"])
        self.replay_c = lambda: lib.gdn_replay_accepted(ra, par, acc, s)

    def h2d(self):
        self.packed.copy_(self.host, non_blocking=True)
        return self.host.numel()

    def d2h(self):
        self.o_host.copy_(self.o, non_blocking=True)
        return self.o.numel() * 4


def run_ours(args, wl_name, world, rank, local):
    import torch

    import hybrid_gated_deltanet_delta_gb300 as gdn

    torch.cuda.set_device(local)
    gdn.load()
    wl = WORKLOADS[wl_name]
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    if wl_name == "prefill8192":
        return run_prefill(args, gdn, torch, flush, world, rank, local)

    Hk, Hv, dk, dv = HEADS["Hk"], HEADS["Hv"], HEADS["dk"], HEADS["dv"]
    B, N = wl["B"], wl["N"]
    replay = wl.get("replay", False)
    index = wl.get("index", False)
    snap16 = wl.get("snap16", False)
    batched = wl_name.startswith("batched8x16")
    L = args.layers if (args.layers and batched) else wl["layers"]
    vbytes = verify_bytes(B, N, Hk, Hv, dk, dv, tree=wl.get("tree", False), persist=not replay,
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
            ws.layers = [VerifyCase(synthetic.batched8x16_layer(l), torch, pinned=True,
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
            inp = synthetic.tree22() if wl.get("tree") else synthetic.chain16()
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
        if index:
            gdn.gdn_commit_index(ws.accept, ws.slot_idx, N=N)
            return
        if replay:
            # checkpoint and replay: the accepted prefix of every layer again
            for c in ws.layers:
                c.replay(gdn)
            return
        gdn.gdn_commit_accepted(ws.snap_all, ws.accept, ws.cache_all, B=B, N=N, Hv=Hv, dk=dk,
                                dv=dv, n_layers=len(ws.layers),
                                snap_layer_stride=B * N * Hv * dk * dv,
                                cache_layer_stride=B * Hv * dk * dv, slot=ws.slot, n_slots=B)

    def step(ws, ev=None):
        """verify every layer, then commit, through the binding's functions;
        ev = (start, after_verify, end) events."""
        if ev is not None:
            ev[0].record(stream)
        for c in ws.layers:
            c.verify(gdn)
        if ev is not None:
            ev[1].record(stream)
        commit(ws)
        if ev is not None:
            ev[2].record(stream)

    def bind_set(ws):
        """The set's step as pre-marshalled C-ABI calls (see VerifyCase.bind)."""
        import ctypes

        lib = gdn.load()
        s = ctypes.c_void_p(stream.cuda_stream)
        for c in ws.layers:
            c.bind(gdn, stream)
        if index:
            acc, sl = ctypes.c_void_p(ws.accept.data_ptr()), ctypes.c_void_p(ws.slot_idx.data_ptr())
            ws.commit_c = [lambda: lib.gdn_commit_index(acc, B, N, 0, sl, None, s)]
        elif replay:
            ws.commit_c = [c.replay_c for c in ws.layers]
        else:
            fn = lib.gdn_commit_accepted_f16 if snap16 else lib.gdn_commit_accepted
            cargs = (ctypes.c_void_p(ws.snap_all.data_ptr()), B * N * Hv * dk * dv,
                     ctypes.c_void_p(ws.accept.data_ptr()),
                     ctypes.c_void_p(ws.cache_all.data_ptr()), Hv * dk * dv, B * Hv * dk * dv,
                     ctypes.c_void_p(ws.slot.data_ptr()), B, B, N, Hv, dk, dv,
                     len(ws.layers), None, s)
            ws.commit_c = [lambda: fn(*cargs)]
        ws.verify_c = [c.verify_c for c in ws.layers]

    def step_c(ws, ev=None):
        """step() through the pre-marshalled calls; any non-zero status raises."""
        if ev is not None:
            ev[0].record(stream)
        for f in ws.verify_c:
            if f():
                raise RuntimeError("verify launch failed")
        if ev is not None:
            ev[1].record(stream)
        for f in ws.commit_c:
            if f():
                raise RuntimeError("commit launch failed")
        if ev is not None:
            ev[2].record(stream)

    sets = [make_set() for _ in range(n_sets)]
    for ws in sets:
        bind_set(ws)
    layers = sets[0].layers
    launches_per_step = len(layers) * 2 if replay else len(layers) + 1
    n_warm = max(args.warmup, n_sets)
    for i in range(n_warm):  # the binding's own functions, then the bound calls
        step(sets[i % n_sets])
    th = time.perf_counter()
    for i in range(n_warm):
        if flush_each:
            flush.fill_(1.0)
        step_c(sets[i % n_sets])
    host_s = (time.perf_counter() - th) / n_warm
    torch.cuda.synchronize()

    gpu_id = gpu_uuid(torch, local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.25)
    barrier(world)
    if not flush_each:
        flush.fill_(0.0)  # the first timed step starts from an L2 without its data
    torch.cuda.synchronize()
    t0 = time.time()
    hold_device(torch, host_s, args.steps)
    if flush_each:
        # the flush between steps is excluded: one event pair per step phase
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(float(i))
            step_c(sets[i % n_sets], evs[i])
        torch.cuda.synchronize()
        step_ms = [e[0].elapsed_time(e[2]) for e in evs]
        verify_ms = [e[0].elapsed_time(e[1]) / len(layers) for e in evs]
        total_ms = sum(step_ms)
    else:
        # back-to-back steps between one event pair, as a serving loop issues them
        e_run = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e_run[0].record(stream)
        for i in range(args.steps):
            step_c(sets[i % n_sets])
        e_run[1].record(stream)
        torch.cuda.synchronize()
        total_ms = e_run[0].elapsed_time(e_run[1])
        step_ms = None
        # the dominant kernel on its own: verify launches back to back over the
        # same rotating copies (every launch again misses L2), one event pair
        k_roof = min(args.steps, 1000)
        hold_device(torch, host_s, k_roof)
        e_roof = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e_roof[0].record(stream)
        for i in range(k_roof):
            for f in sets[i % n_sets].verify_c:
                if f():
                    raise RuntimeError("verify launch failed")
        e_roof[1].record(stream)
        torch.cuda.synchronize()
        verify_ms = [e_roof[0].elapsed_time(e_roof[1]) / (k_roof * len(layers))]
    barrier(world)
    t1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    total_ms = max_over_ranks(total_ms, world)

    # end to end through the public API: host inputs -> device -> verify/commit -> host o
    for ws in sets:
        if ws.cache_init is not None:
            ws.cache_all.copy_(ws.cache_init)
    e2e_steps = min(args.steps, 200)
    e2e_s = 0.0
    h2d = d2h = 0
    for i in range(e2e_steps + 3):
        ws = sets[i % n_sets]
        flush.fill_(float(i))
        torch.cuda.synchronize()
        ta = time.perf_counter()
        h2d = sum(c.h2d() for c in ws.layers)
        step(ws)
        d2h = sum(c.d2h() for c in ws.layers)
        torch.cuda.synchronize()
        if i >= 3:
            e2e_s += time.perf_counter() - ta
    e2e_s = max_over_ranks(e2e_s, world)

    node_heads = B * N * Hv * len(layers)
    value = job_throughput(node_heads, args.steps, total_ms, world)
    hbm, bf16, peak_kind = measured_peaks()
    launch_ms = statistics.mean(verify_ms)
    achieved = vbytes / (launch_ms / 1e3) / 1e9
    clocks = sampler.summary(t0, t1)
    if rank != 0:
        return None
    return {
        "metric": METRIC,
        "value": value,
        "unit": "node-heads/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
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
                       "CUDA events on the launch stream around the K back-to-back steps; the "
                       "verify kernel alone from a second back-to-back run of verify launches"),
            "launch": "programmatic dependent launch (each kernel waits on its predecessor "
                      "before any global-memory access)",
            "parallelism": f"replicas x{world}, no collective",
            "verify_ms_per_launch": launch_ms,
            **({"step_ms_p10": float(np.percentile(step_ms, 10)),
                "step_ms_p90": float(np.percentile(step_ms, 90))} if step_ms else {}),
        },
        "roofline": {
            "bound": "hbm",
            "kernel": ("gdn_verify_tree" if wl.get("tree") else "gdn_verify_chain") +
                      (" (no snapshots)" if replay else
                       " (binary16 snapshots)" if wl.get("snap16") else
                       " (state and snapshots in the slot region)" if index else ""),
            "achieved": achieved,
            "peak": hbm,
            "unit": "GB/s",
            "frac": achieved / hbm,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind ==
            "measured" else "fallback 6.8 TB/s",
            "algorithmic_bytes_per_launch": vbytes,
            "traffic": profiled_traffic("verify", wl_name),
        },
        "e2e": {
            "value": world * node_heads * e2e_steps / e2e_s,
            "unit": "node-heads/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
        },
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }


def run_prefill(args, gdn, torch, flush, world, rank, local):
    inp = synthetic.prefill8192()
    T, Hk, Hv, dk, dv = inp["T"], inp["Hk"], inp["Hv"], inp["dk"], inp["dv"]
    q, k, v = (_dev(inp[n], torch) for n in ("q", "k", "v"))
    alpha, beta = _dev(inp["alpha"], torch), _dev(inp["beta"], torch)
    state0 = _dev(inp["state"], torch)
    state = state0.clone()
    o = torch.empty((T, Hv, dv), device="cuda")
    wbytes = gdn.gdn_prefill_workspace_bytes(T, Hk, Hv, dk, dv, 64)
    ws = torch.empty(max(wbytes, 16), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step(ev=None):
        state.copy_(state0)
        if ev is not None:
            ev[0].record(stream)
        gdn.gdn_prefill_chunked(q, k, v, alpha, beta, state, o, ws)
        if ev is not None:
            ev[1].record(stream)

    th = time.perf_counter()
    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    host_s = (time.perf_counter() - th) / max(1, args.warmup)
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid(torch, local))
    sampler.start()
    time.sleep(0.25)
    steps = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    hold_device(torch, host_s, steps)
    for i in range(steps):
        flush.fill_(float(i))
        step(evs[i])
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    ms = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = max_over_ranks(sum(ms), world)
    # end to end: host inputs (pinned) -> device -> prefill -> host o and state
    hq, hk, hv, ha, hb = (x.cpu().pin_memory() for x in (q, k, v, alpha, beta))
    hs0 = state0.cpu().pin_memory()
    ho = torch.empty(o.shape).pin_memory()
    hst = torch.empty(state.shape).pin_memory()
    e2e_steps = min(steps, 20)
    e2e_s = 0.0
    for i in range(e2e_steps + 2):
        flush.fill_(float(i))
        torch.cuda.synchronize()
        ta = time.perf_counter()
        for d, h in ((q, hq), (k, hk), (v, hv), (alpha, ha), (beta, hb), (state, hs0)):
            d.copy_(h, non_blocking=True)
        gdn.gdn_prefill_chunked(q, k, v, alpha, beta, state, o, ws)
        ho.copy_(o, non_blocking=True)
        hst.copy_(state, non_blocking=True)
        torch.cuda.synchronize()
        if i >= 2:
            e2e_s += time.perf_counter() - ta
    e2e_s = max_over_ranks(e2e_s, world)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, ha, hb, hs0))
    d2h = ho.numel() * 4 + hst.numel() * 4
    hbm, bf16, kind = measured_peaks()
    pbytes = prefill_bytes(T, Hk, Hv, dk, dv)
    launch_ms = statistics.mean(ms)
    gbs = pbytes / (launch_ms / 1e3) / 1e9
    flops = prefill_flops(T, Hk, Hv, dk, dv)
    tflops = flops / (launch_ms / 1e3) / 1e12
    if rank != 0:
        return None
    return {
        "metric": METRIC,
        "value": world * T * Hv * steps / (total_ms / 1e3),
        "unit": "token-heads/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": total_ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"prefill8192: {WORKLOADS['prefill8192']['desc']}",
                   "T": T, "Hk": Hk, "Hv": Hv, "dk": dk, "dv": dv, "chunk": 64,
                   "l2": "flushed by a 256 MiB write before every step; flush not timed",
                   "timing": "CUDA events around each prefill call (prep + scan kernels) "
                             "on the launch stream",
                   "hbm_achieved_gbs": gbs, "hbm_frac_of_measured": gbs / hbm,
                   "algorithmic_bytes_per_call": pbytes},
        "roofline": {"bound": "tensor", "kernel": "gdn_prefill_chunked (prep + scan)",
                     "achieved": tflops, "peak": bf16, "unit": "TFLOP/s", "frac": tflops / bf16,
                     "peak_source": kind, "algorithmic_flops_per_launch": flops,
                     "traffic": profiled_traffic("prefill", "prefill8192")},
        "e2e": {"value": world * T * Hv * e2e_steps / e2e_s, "unit": "token-heads/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * steps,   # prep + scan per call
        "clocks": sampler.summary(t0, t1),
    }


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
    if rank != 0:
        return None
    if wl_name == "prefill8192":
        for _ in range(args.warmup):
            oracle_step_sample(wl_name, 1)
        spent, done = 0.0, 0
        for _ in range(args.steps):
            dt, n = oracle_step_sample(wl_name, 1)
            spent += dt
            done += n
        unit, sample = "token-heads/s", "8192 tokens x 1 value head per step (step form)"
    else:
        smp = OracleSampler(wl_name)
        for _ in range(args.warmup):
            smp.run(1)
        done = 0
        t0 = time.perf_counter()
        for _ in range(args.steps):
            done += smp.run(1)
        spent = time.perf_counter() - t0
        unit = "node-heads/s"
        sample = f"verify + commit of 1 value head x {smp.inp['N']} nodes per step"
    value = done / spent
    wl = WORKLOADS[wl_name]
    return {
        "metric": METRIC, "value": value, "unit": unit, "impl": "reference",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * spent / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl_name}: {wl['desc']}"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="chain16", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0,
                    help="batched8x16 only: run this many of the 48 layers (profiling slices)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (for quick runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        out = run_reference(args, args.workload, world, rank)
    else:
        out = run_ours(args, args.workload, world, rank, local)
        if out is not None:
            out["cpu_baseline"] = (None if args.no_cpu_baseline or world > 1 else
                                   cpu_baseline(args.workload))
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
