"""Seeded synthetic inputs for the gated delta-rule verify / commit / prefill path.

This module is shared by the CPU oracle's tests, the CUDA path's tests and the
benchmark.  It only draws random numbers and shapes them (normal draws, the
per-head L2 normalisation and bf16 rounding that the workloads prescribe for
q/k, the alpha/beta gate transforms, random trees and accept indices).  It
holds none of the recurrence's arithmetic.

Workloads (all synthetic; the pages measure on GSM8K / HumanEval / essays with
trained weights, none of which is available here, so projected activations of
the same shapes and distributions stand in for them):

  tiny_chain      B=1, Hk=Hv=2, d=16, chain of 4, fp32 everything
  chain16         B=1, Hk=16, Hv=48, d=128, chain of 16, bf16 q/k/v
  tree22          B=1, Hk=16, Hv=48, d=128, DDTree of 22 nodes, bf16 q/k/v
  batched8x16     B=8, chain of 16, same heads, 48 layers with fresh inputs
  prefill8192     T=8192, Hk=16, Hv=48, d=128, chunk 64, bf16 q/k/v

Distributions: q, k ~ N(0,1) then L2-normalised per (node, head) in float64
and rounded to bf16 (round-to-nearest-even); v ~ N(0,1) rounded to bf16;
beta = sigmoid(z); alpha = exp(-softplus(z)) for tiny_chain and
alpha = 0.9 + 0.1 * exp(-softplus(z)) in (0.9, 1) for the rest; initial
state ~ N(0, sigma) with sigma = 0.1 (tiny_chain) or 0.05; z ~ N(0,1).
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 0x6D6E0000
GOLDEN_RATIO_64 = 0x9E3779B97F4A7C15
MASK64 = (1 << 64) - 1

WORKLOADS = ("tiny_chain", "chain16", "tree22", "batched8x16", "prefill8192", "batched8x22")


def workload_seed(name: str) -> int:
    return SEED_BASE + WORKLOADS.index(name)


def layer_seed(base: int, layer: int) -> int:
    return (base ^ (((layer + 1) * GOLDEN_RATIO_64) & MASK64)) & MASK64


# ---------------------------------------------------------------- bf16 helpers
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((b >> 16) & 1) + 0x7FFF
    return ((b + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _l2_normalise(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / n


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def _softplus(z):
    return np.log1p(np.exp(-np.abs(z))) + np.maximum(z, 0.0)


def _alpha(z: np.ndarray, kind: str) -> np.ndarray:
    decay = np.exp(-_softplus(z))  # in (0, 1)
    if kind == "unit":
        return decay
    if kind == "near_one":
        return 0.9 + 0.1 * decay
    raise ValueError(kind)


def random_tree(rng: np.random.Generator, n: int, depth_cap: int = 16) -> np.ndarray:
    """parent[0] = -1; node i > 0 picks a parent uniformly among earlier nodes
    whose depth is below the cap (root depth is 1)."""
    parent = np.full(n, -1, dtype=np.int32)
    depth = np.zeros(n, dtype=np.int64)
    depth[0] = 1
    for i in range(1, n):
        cand = np.nonzero(depth[:i] < depth_cap)[0]
        p = int(cand[rng.integers(0, len(cand))])
        parent[i] = p
        depth[i] = depth[p] + 1
    return parent


def _cast(x64: np.ndarray, dtype: str):
    """Return (stored array, exact float64 view of the stored values)."""
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x64.astype(np.float32))
        return bits, bf16_bits_to_f32(bits).astype(np.float64)
    if dtype == "f32":
        x32 = x64.astype(np.float32)
        return x32, x32.astype(np.float64)
    raise ValueError(dtype)


def make_verify_inputs(*, B, N, Hk, Hv, dk, dv, dtype, alpha_kind, state_sigma, seed,
                       tree=False, n_slots=None, depth_cap=16, slot_perm=True):
    """One verify block for B sequences.

    Returns a dict of numpy arrays in the device layouts:
      q, k      [B][N][Hk][dk]   bf16 bits (uint16) or float32
      v         [B][N][Hv][dv]   same dtype
      alpha     [B][N][Hv]       float32
      beta      [B][N][Hv]       float32
      cache     [n_slots][Hv][dk][dv] float32 (recurrent-state cache)
      slot      [B] int32        (a permutation of the first B slots)
      parent    [B][N] int32     (tree only; chain => i-1)
      accept    [B] int32        accepted node index (chain: L-1, L in [1,N])
    plus *_f64 exact float64 copies of q, k, v for the oracle.
    """
    rng = np.random.default_rng(seed)
    if n_slots is None:
        n_slots = B
    q = _l2_normalise(rng.standard_normal((B, N, Hk, dk)))
    k = _l2_normalise(rng.standard_normal((B, N, Hk, dk)))
    v = rng.standard_normal((B, N, Hv, dv))
    q_s, q64 = _cast(q, dtype)
    k_s, k64 = _cast(k, dtype)
    v_s, v64 = _cast(v, dtype)
    alpha = _alpha(rng.standard_normal((B, N, Hv)), alpha_kind).astype(np.float32)
    beta = _sigmoid(rng.standard_normal((B, N, Hv))).astype(np.float32)
    cache = (rng.standard_normal((n_slots, Hv, dk, dv)) * state_sigma).astype(np.float32)
    slot = (rng.permutation(n_slots)[:B] if slot_perm else np.arange(B)).astype(np.int32)
    if tree:
        parent = np.stack([random_tree(rng, N, depth_cap) for _ in range(B)]).astype(np.int32)
        accept = rng.integers(0, N, size=B).astype(np.int32)
    else:
        parent = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
        accept = (rng.integers(1, N + 1, size=B) - 1).astype(np.int32)
    return dict(q=q_s, k=k_s, v=v_s, q_f64=q64, k_f64=k64, v_f64=v64,
                alpha=alpha, beta=beta, cache=cache, slot=slot, parent=parent,
                accept=accept, B=B, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv,
                dtype=dtype, n_slots=n_slots, tree=tree)


def make_prefill_inputs(*, T, Hk, Hv, dk, dv, dtype, alpha_kind, state_sigma, seed):
    """One prefill sequence: q,k [T][Hk][dk], v [T][Hv][dv], alpha/beta [T][Hv],
    initial state [Hv][dk][dv] float32."""
    rng = np.random.default_rng(seed)
    q = _l2_normalise(rng.standard_normal((T, Hk, dk)))
    k = _l2_normalise(rng.standard_normal((T, Hk, dk)))
    v = rng.standard_normal((T, Hv, dv))
    q_s, q64 = _cast(q, dtype)
    k_s, k64 = _cast(k, dtype)
    v_s, v64 = _cast(v, dtype)
    alpha = _alpha(rng.standard_normal((T, Hv)), alpha_kind).astype(np.float32)
    beta = _sigmoid(rng.standard_normal((T, Hv))).astype(np.float32)
    state = (rng.standard_normal((Hv, dk, dv)) * state_sigma).astype(np.float32)
    return dict(q=q_s, k=k_s, v=v_s, q_f64=q64, k_f64=k64, v_f64=v64,
                alpha=alpha, beta=beta, state=state, T=T, Hk=Hk, Hv=Hv,
                dk=dk, dv=dv, dtype=dtype)


# --------------------------------------------------------------- the workloads
HEADS = dict(Hk=16, Hv=48, dk=128, dv=128)


def tiny_chain(seed=None):
    return make_verify_inputs(B=1, N=4, Hk=2, Hv=2, dk=16, dv=16, dtype="f32",
                              alpha_kind="unit", state_sigma=0.1,
                              seed=workload_seed("tiny_chain") if seed is None else seed)


def tiny_chain_accept() -> int:
    """The tiny chain commits node 2 (accept length 3)."""
    return 2


def chain16(seed=None, B=1):
    return make_verify_inputs(B=B, N=16, dtype="bf16", alpha_kind="near_one", state_sigma=0.05,
                              seed=workload_seed("chain16") if seed is None else seed, **HEADS)


def tree22(seed=None, B=1):
    return make_verify_inputs(B=B, N=22, dtype="bf16", alpha_kind="near_one", state_sigma=0.05,
                              tree=True, seed=workload_seed("tree22") if seed is None else seed,
                              **HEADS)


def batched8x16_layer(layer: int):
    """Inputs of one of the 48 layers.  The slot of each sequence and its
    accept index belong to the batch, not the layer, so they are drawn once
    from the workload's base seed and shared by every layer."""
    base = workload_seed("batched8x16")
    inp = make_verify_inputs(B=8, N=16, dtype="bf16", alpha_kind="near_one", state_sigma=0.05,
                             seed=layer_seed(base, layer), **HEADS)
    rng = np.random.default_rng(base)
    inp["slot"] = rng.permutation(8).astype(np.int32)
    inp["accept"] = (rng.integers(1, 17, size=8) - 1).astype(np.int32)
    return inp


def batched8x22_layer(layer: int):
    """One of the 48 layers of a batch of 8 sequences, each verifying a
    22-node draft tree.  The trees, slots and accepted nodes belong to the
    batch (every layer verifies the same trees), so they are drawn once from
    the workload's base seed; q, k, v, gates and states are per layer."""
    base = workload_seed("batched8x22")
    inp = make_verify_inputs(B=8, N=22, dtype="bf16", alpha_kind="near_one", state_sigma=0.05,
                             tree=True, seed=layer_seed(base, layer), **HEADS)
    rng = np.random.default_rng(base)
    inp["slot"] = rng.permutation(8).astype(np.int32)
    inp["parent"] = np.stack([random_tree(rng, 22) for _ in range(8)]).astype(np.int32)
    inp["accept"] = rng.integers(0, 22, size=8).astype(np.int32)
    return inp


BATCHED_LAYERS = 48


def prefill8192(seed=None, T=8192):
    return make_prefill_inputs(T=T, dtype="bf16", alpha_kind="near_one", state_sigma=0.05,
                               seed=workload_seed("prefill8192") if seed is None else seed,
                               **HEADS)
