"""CPU oracle for the gated delta-rule verify / commit / prefill path.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline import this package.  The CUDA library never does, and this package
never imports the library.  The arithmetic lives in gdn_oracle.cpp (plain C++,
float64 or long double); this file builds it with g++ and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

OK = 0
ERR_INVALID_ARG = -1
ERR_BAD_TREE = -5
ERR_ACCEPT_RANGE = -6
ERR_SLOT_RANGE = -7


def build(force: bool = False) -> str:
    """Compile gdn_oracle.cpp into liboracle.so (no fast-math, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared",
                               "-fno-fast-math", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def bind(lib):
    """Declare the C signatures on a loaded oracle library and return it."""
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    for name in ("oracle_verify_f64", "oracle_verify_ld"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [P, P, P, P, P, P, i64, P, i32, P, i32, i32, i32, i32, i32, i32, P, P,
                      i32]
    lib.oracle_tree_depth.restype = ctypes.c_int
    lib.oracle_tree_depth.argtypes = [P, i32, i32, P, i32]
    lib.oracle_commit_f64.restype = ctypes.c_int
    lib.oracle_commit_f64.argtypes = [P, i64, P, P, i64, i64, P, i32, i32, i32, i32, i32,
                                      i32, i32]
    lib.oracle_prepare_inputs_f64.restype = ctypes.c_int
    lib.oracle_prepare_inputs_f64.argtypes = [P, P, i64, i32, P, P, i64]
    lib.oracle_conv_commit_f64.restype = ctypes.c_int
    lib.oracle_conv_commit_f64.argtypes = [P, P, i64, P, i32, P, P, i32, i32, i32, i32]
    lib.oracle_commit_index.restype = ctypes.c_int
    lib.oracle_commit_index.argtypes = [P, i32, i32, i32, P]
    lib.oracle_replay_f64.restype = ctypes.c_int
    lib.oracle_replay_f64.argtypes = [P, P, P, P, P, i64, P, i32, P, P, i32, i32, i32, i32, i32,
                                      i32]
    lib.oracle_prefill_step_f64.restype = ctypes.c_int
    lib.oracle_prefill_step_f64.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                            i32, P, P]
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = bind(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def verify(q, k, v, alpha, beta, cache, slot, parent, *, B, N, Hk, Hv, dk, dv,
           cache_slot_stride=None, n_slots=None, precision="f64", max_depth=0):
    """Run a verify block.  parent=None -> chain.  Returns (status, snap, o)
    with snap [B][N][Hv][dk][dv] and o [B][N][Hv][dv] in the chosen precision.
    max_depth > 0 rejects (skips) a tree with a node deeper than that."""
    lib = _load()
    R = np.float64 if precision == "f64" else np.longdouble
    fn = lib.oracle_verify_f64 if precision == "f64" else lib.oracle_verify_ld
    cache = _c(cache, R)
    if cache_slot_stride is None:
        cache_slot_stride = Hv * dk * dv
    if n_slots is None:
        n_slots = cache.size // cache_slot_stride
    snap = np.zeros((B, N, Hv, dk, dv), dtype=R)
    o = np.zeros((B, N, Hv, dv), dtype=R)
    arrs = [_c(q, R), _c(k, R), _c(v, R), _c(alpha, R), _c(beta, R)]
    slot_a = None if slot is None else _c(slot, np.int32)
    par_a = None if parent is None else _c(parent, np.int32)
    st = fn(*[_ptr(a) for a in arrs], _ptr(cache), cache_slot_stride, _ptr(slot_a), n_slots,
            _ptr(par_a), B, N, Hk, Hv, dk, dv, _ptr(snap), _ptr(o), max_depth)
    return st, snap, o


def verify_inputs(inp, tree=None, precision="f64"):
    """verify() on a dict made by synthetic.make_verify_inputs."""
    tree = inp["tree"] if tree is None else tree
    return verify(inp["q_f64"], inp["k_f64"], inp["v_f64"], inp["alpha"], inp["beta"],
                  inp["cache"], inp["slot"], inp["parent"] if tree else None, B=inp["B"],
                  N=inp["N"], Hk=inp["Hk"], Hv=inp["Hv"], dk=inp["dk"], dv=inp["dv"],
                  n_slots=inp["n_slots"], precision=precision)


def tree_depth(parent, max_depth=0):
    lib = _load()
    parent = _c(parent, np.int32)
    B, N = parent.shape
    depth = np.zeros((B, N), dtype=np.int32)
    st = lib.oracle_tree_depth(_ptr(parent), B, N, _ptr(depth), max_depth)
    return st, depth


def commit(snap, accept, cache, slot, *, B, N, Hv, dk, dv, n_layers=1,
           snap_layer_stride=0, cache_slot_stride=None, cache_layer_stride=0, n_slots=None):
    """In-place copy of the accepted snapshots into `cache` (float64 array)."""
    lib = _load()
    assert cache.dtype == np.float64 and cache.flags.c_contiguous
    snap = _c(snap, np.float64)
    if cache_slot_stride is None:
        cache_slot_stride = Hv * dk * dv
    if n_slots is None:
        n_slots = (cache.size - (n_layers - 1) * cache_layer_stride) // cache_slot_stride
    acc = _c(accept, np.int32)
    slot_a = None if slot is None else _c(slot, np.int32)
    return lib.oracle_commit_f64(_ptr(snap), snap_layer_stride, _ptr(acc), _ptr(cache),
                                 cache_slot_stride, cache_layer_stride, _ptr(slot_a), n_slots,
                                 B, N, Hv, dk, dv, n_layers)


def prepare_inputs(q, k, a, b):
    """Raw projections -> verify inputs (float64 copies): q, k L2-normalised
    over their last axis, alpha = exp(-softplus(a)), beta = sigmoid(b)."""
    lib = _load()
    q = np.array(q, dtype=np.float64, order="C")
    k = np.array(k, dtype=np.float64, order="C")
    al = np.array(a, dtype=np.float64, order="C")
    be = np.array(b, dtype=np.float64, order="C")
    assert q.shape == k.shape and al.shape == be.shape
    d = q.shape[-1]
    st = lib.oracle_prepare_inputs_f64(_ptr(q), _ptr(k), q.size // d, d, _ptr(al), _ptr(be),
                                       al.size)
    assert st == OK
    return q, k, al, be


def conv_commit(x, state, slot, parent, accept, *, n_slots=None):
    """Convolution-history commit in place on `state` [n_slots, C, W] (float64);
    x [B, N, C].  parent=None -> chain.  Returns the status."""
    lib = _load()
    assert state.dtype == np.float64 and state.flags.c_contiguous
    x = _c(x, np.float64)
    B, N, C = x.shape
    W = state.shape[-1]
    if n_slots is None:
        n_slots = state.shape[0]
    slot_a = None if slot is None else _c(slot, np.int32)
    par_a = None if parent is None else _c(parent, np.int32)
    return lib.oracle_conv_commit_f64(_ptr(x), _ptr(state), C * W, _ptr(slot_a), n_slots,
                                      _ptr(par_a), _ptr(_c(accept, np.int32)), B, N, C, W)


def commit_index(accept, slot, *, N, base=0):
    """Index-table commit in place on `slot` (int32 array of B entries)."""
    lib = _load()
    assert slot.dtype == np.int32 and slot.flags.c_contiguous
    acc = _c(accept, np.int32)
    return lib.oracle_commit_index(_ptr(acc), len(acc), N, base, _ptr(slot))


def replay(k, v, alpha, beta, cache, slot, parent, accept, *, B, N, Hk, Hv, dk, dv,
           cache_slot_stride=None, n_slots=None):
    """Replay commit in place on `cache` (float64 array): the recurrence over
    each sequence's accepted path from its cached state.  parent=None -> chain
    (accept = accept length - 1).  Returns the status."""
    lib = _load()
    assert cache.dtype == np.float64 and cache.flags.c_contiguous
    if cache_slot_stride is None:
        cache_slot_stride = Hv * dk * dv
    if n_slots is None:
        n_slots = cache.size // cache_slot_stride
    arrs = [_c(k, np.float64), _c(v, np.float64), _c(alpha, np.float64), _c(beta, np.float64)]
    slot_a = None if slot is None else _c(slot, np.int32)
    par_a = None if parent is None else _c(parent, np.int32)
    acc = _c(accept, np.int32)
    return lib.oracle_replay_f64(*[_ptr(a) for a in arrs], _ptr(cache), cache_slot_stride,
                                 _ptr(slot_a), n_slots, _ptr(par_a), _ptr(acc), B, N, Hk, Hv,
                                 dk, dv)


def prefill_step(q, k, v, alpha, beta, state, *, T, Hk, Hv, dk, dv, heads=None):
    """Token-by-token recurrence.  Returns (status, final_state, o); heads=(h0, nh)
    restricts the work to value heads h0..h0+nh-1 (others left as given / zero)."""
    lib = _load()
    h0, nh = (0, Hv) if heads is None else heads
    st_arr = _c(state, np.float64).copy()
    o = np.zeros((T, Hv, dv), dtype=np.float64)
    arrs = [_c(q, np.float64), _c(k, np.float64), _c(v, np.float64), _c(alpha, np.float64),
            _c(beta, np.float64)]
    st = lib.oracle_prefill_step_f64(*[_ptr(a) for a in arrs], T, Hk, Hv, dk, dv, h0, nh,
                                     _ptr(st_arr), _ptr(o))
    return st, st_arr, o
