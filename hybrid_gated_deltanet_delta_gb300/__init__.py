"""GB300 gated delta-rule verification library: Python binding.

A thin ctypes layer over libgdn.so (C ABI in include/gdn.h).  It only
marshals arguments: torch tensors in, raw device pointers and sizes out, the
current torch CUDA stream as the launch stream.  Every step of the path runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and the
functions raise if the library is missing or a call fails.

Entry points (same names as the C ABI):
  gdn_verify_chain, gdn_verify_chain_f16, gdn_verify_tree, gdn_verify_tree_f16,
  gdn_commit_accepted,
  gdn_commit_accepted_f16, gdn_commit_index, gdn_conv_commit,
  gdn_replay_accepted,
  gdn_prefill_chunked, gdn_prefill_workspace_bytes, gdn_prefill_chunked_noalloc
and, for serving loops that issue the same call every step, bound calls
(bind_verify_chain, bind_verify_tree, bind_commit_accepted,
bind_replay_accepted, bind_prefill_chunked): the arguments are marshalled once
and each call is one ctypes call.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID_ARG = -1
GDN_ERR_UNSUPPORTED = -2
GDN_ERR_MISALIGNED = -3
GDN_ERR_CUDA = -4
GDN_ERR_BAD_TREE = -5
GDN_ERR_ACCEPT_RANGE = -6
GDN_ERR_SLOT_RANGE = -7
GDN_ERR_WORKSPACE = -8
GDN_ERR_SCRATCH_LIMIT = -9
GDN_ERR_TIMEOUT = -10
PREFILL_NOALLOC_SCRATCH_BYTES = 16 << 20

GDN_F32 = 0
GDN_BF16 = 1

_lib = None


class GdnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


class VerifyArgs(ctypes.Structure):
    """Mirror of gdn_verify_args."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("alpha", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("state_cache", ctypes.c_void_p), ("slot", ctypes.c_void_p),
        ("snapshots", ctypes.c_void_p), ("o", ctypes.c_void_p), ("status", ctypes.c_void_p),
        ("cache_slot_stride", ctypes.c_int64), ("n_slots", ctypes.c_int32),
        ("B", ctypes.c_int32), ("N", ctypes.c_int32), ("Hk", ctypes.c_int32),
        ("Hv", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
        ("in_dtype", ctypes.c_int32), ("tile_cols", ctypes.c_int32),
        ("row_warps", ctypes.c_int32), ("max_depth", ctypes.c_int32),
    ]


def load(path: str | None = None):
    """Load libgdn.so (built by __graft_entry__.build()); raise if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libgdn.so not found at {p}: build it first "
                           "(python -m hybrid_gated_deltanet_delta_gb300.build)")
    lib = ctypes.CDLL(p)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.gdn_verify_chain.argtypes = [ctypes.POINTER(VerifyArgs), P]
    lib.gdn_verify_chain.restype = ctypes.c_int
    lib.gdn_verify_tree.argtypes = [ctypes.POINTER(VerifyArgs), P, P, P]
    lib.gdn_verify_tree.restype = ctypes.c_int
    lib.gdn_commit_accepted.argtypes = [P, i64, P, P, i64, i64, P, i32, i32, i32, i32, i32, i32,
                                        i32, P, P]
    lib.gdn_commit_accepted.restype = ctypes.c_int
    lib.gdn_verify_chain_prep.argtypes = [ctypes.POINTER(VerifyArgs), P]
    lib.gdn_verify_chain_prep.restype = ctypes.c_int
    lib.gdn_verify_tree_prep.argtypes = [ctypes.POINTER(VerifyArgs), P, P, P]
    lib.gdn_verify_tree_prep.restype = ctypes.c_int
    lib.gdn_replay_accepted_prep.argtypes = [ctypes.POINTER(VerifyArgs), P, P, P]
    lib.gdn_replay_accepted_prep.restype = ctypes.c_int
    lib.gdn_verify_chain_f16.argtypes = [ctypes.POINTER(VerifyArgs), P, P]
    lib.gdn_verify_chain_f16.restype = ctypes.c_int
    lib.gdn_verify_tree_f16.argtypes = [ctypes.POINTER(VerifyArgs), P, P, P, P]
    lib.gdn_verify_tree_f16.restype = ctypes.c_int
    lib.gdn_commit_accepted_f16.argtypes = [P, i64, P, P, i64, i64, P, i32, i32, i32, i32, i32,
                                            i32, i32, P, P]
    lib.gdn_commit_accepted_f16.restype = ctypes.c_int
    lib.gdn_conv_commit.argtypes = [P, i32, P, i64, P, i32, P, P, i32, i32, i32, i32, P, P]
    lib.gdn_conv_commit.restype = ctypes.c_int
    lib.gdn_commit_index.argtypes = [P, i32, i32, i32, P, P, P]
    lib.gdn_commit_index.restype = ctypes.c_int
    lib.gdn_replay_accepted.argtypes = [ctypes.POINTER(VerifyArgs), P, P, P]
    lib.gdn_replay_accepted.restype = ctypes.c_int
    lib.gdn_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.gdn_prefill_workspace_bytes.restype = sz
    lib.gdn_prefill_chunked.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32, P, P,
                                        P, sz, P, P]
    lib.gdn_prefill_chunked.restype = ctypes.c_int
    lib.gdn_prefill_chunked_noalloc.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32,
                                                P, P, P, P]
    lib.gdn_prefill_chunked_noalloc.restype = ctypes.c_int
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_version.argtypes = []
    lib.gdn_version.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load().gdn_status_string(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


# ------------------------------------------------------------- marshalling
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code, where):
    if code != GDN_OK:
        raise GdnError(code, where)


def _dtype_code(t):
    import torch

    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def make_verify_args(q, k, v, alpha, beta, state_cache, snapshots, o, *, slot=None, n_slots=None,
                     status=None, cache_slot_stride=None, tile_cols=0, row_warps=0,
                     max_depth=0):
    """Build a gdn_verify_args from tensors.  q, k [B,N,Hk,dk]; v [B,N,Hv,dv];
    alpha, beta [B,N,Hv] fp32; state_cache [n_slots,Hv,dk,dv] fp32 (or any
    buffer with `cache_slot_stride`); snapshots [B,N,Hv,dk,dv] fp32 or None
    (a chain committed by replay); o [B,N,Hv,dv] fp32.  q and o may be None for
    gdn_replay_accepted."""
    B, N, Hk, dk = k.shape
    Hv, dv = v.shape[2], v.shape[3]
    for t in (q, k, v, alpha, beta, state_cache, snapshots, o):
        _need(t is None or t.is_contiguous(), "all tensors must be contiguous")
    _need((q is None or q.shape == k.shape) and v.shape[:2] == (B, N), "q/k/v shapes disagree")
    _need((q is None or q.dtype == k.dtype) and k.dtype == v.dtype,
          "q, k and v must share a dtype")
    if cache_slot_stride is None:
        cache_slot_stride = Hv * dk * dv
    if n_slots is None:
        n_slots = state_cache.numel() // cache_slot_stride
    def ptr(t):
        return None if t is None else t.data_ptr()

    return VerifyArgs(
        q=ptr(q), k=k.data_ptr(), v=v.data_ptr(), alpha=alpha.data_ptr(),
        beta=beta.data_ptr(), state_cache=state_cache.data_ptr(), slot=ptr(slot),
        snapshots=ptr(snapshots), o=ptr(o), status=ptr(status),
        cache_slot_stride=cache_slot_stride, n_slots=n_slots, B=B, N=N, Hk=Hk, Hv=Hv, dk=dk,
        dv=dv, in_dtype=_dtype_code(k), tile_cols=tile_cols, row_warps=row_warps,
        max_depth=max_depth)


def gdn_verify_chain(q, k, v, alpha, beta, state_cache, snapshots, o, *, slot=None, n_slots=None,
                     status=None, cache_slot_stride=None, tile_cols=0, row_warps=0, stream=None,
                     prep=False):
    """Causal-chain verification; writes snapshots and o (see include/gdn.h).
    prep=True: q, k are raw projections and alpha, beta gate pre-activations
    (gdn_verify_chain_prep)."""
    a = make_verify_args(q, k, v, alpha, beta, state_cache, snapshots, o, slot=slot,
                         n_slots=n_slots, status=status, cache_slot_stride=cache_slot_stride,
                         tile_cols=tile_cols, row_warps=row_warps)
    fn = load().gdn_verify_chain_prep if prep else load().gdn_verify_chain
    _check(fn(ctypes.byref(a), _stream(stream)),
           "gdn_verify_chain_prep" if prep else "gdn_verify_chain")


def gdn_verify_chain_f16(q, k, v, alpha, beta, state_cache, snapshots_f16, o, *, slot=None,
                         n_slots=None, status=None, cache_slot_stride=None, tile_cols=0,
                         row_warps=0, stream=None):
    """Chain verification persisting every node's state as float16 (RNE) in
    snapshots_f16 [B,N,Hv,dk,dv]; outputs unchanged (see include/gdn.h)."""
    import torch

    _need(snapshots_f16.dtype == torch.float16 and snapshots_f16.is_contiguous(),
          "snapshots_f16 must be a contiguous float16 tensor")
    a = make_verify_args(q, k, v, alpha, beta, state_cache, None, o, slot=slot,
                         n_slots=n_slots, status=status, cache_slot_stride=cache_slot_stride,
                         tile_cols=tile_cols, row_warps=row_warps)
    _check(load().gdn_verify_chain_f16(ctypes.byref(a), _ptr(snapshots_f16), _stream(stream)),
           "gdn_verify_chain_f16")


def gdn_verify_tree_f16(q, k, v, alpha, beta, state_cache, snapshots_f16, o, parent, *,
                        depth_out=None, slot=None, n_slots=None, status=None,
                        cache_slot_stride=None, tile_cols=0, row_warps=0, max_depth=0,
                        stream=None):
    """Tree verification persisting every node's state as float16 (RNE) in
    snapshots_f16 [B,N,Hv,dk,dv]; outputs unchanged (see include/gdn.h)."""
    import torch

    _need(snapshots_f16.dtype == torch.float16 and snapshots_f16.is_contiguous(),
          "snapshots_f16 must be a contiguous float16 tensor")
    _need(parent.is_contiguous() and tuple(parent.shape) == tuple(k.shape[:2]),
          "parent must be a contiguous [B,N] int32 tensor")
    a = make_verify_args(q, k, v, alpha, beta, state_cache, None, o, slot=slot,
                         n_slots=n_slots, status=status, cache_slot_stride=cache_slot_stride,
                         tile_cols=tile_cols, row_warps=row_warps, max_depth=max_depth)
    _check(load().gdn_verify_tree_f16(ctypes.byref(a), _ptr(parent), _ptr(depth_out),
                                      _ptr(snapshots_f16), _stream(stream)),
           "gdn_verify_tree_f16")


def gdn_verify_tree(q, k, v, alpha, beta, state_cache, snapshots, o, parent, *, depth_out=None,
                    slot=None, n_slots=None, status=None, cache_slot_stride=None, tile_cols=0,
                    row_warps=0, max_depth=0, stream=None, prep=False):
    """Tree verification; parent [B,N] int32 (see include/gdn.h).  max_depth > 0
    skips (and reports through `status`) any sequence whose tree is deeper.
    prep=True: raw projections and gate pre-activations (gdn_verify_tree_prep)."""
    _need(parent.is_contiguous() and tuple(parent.shape) == tuple(q.shape[:2]),
          "parent must be a contiguous [B,N] int32 tensor")
    a = make_verify_args(q, k, v, alpha, beta, state_cache, snapshots, o, slot=slot,
                         n_slots=n_slots, status=status, cache_slot_stride=cache_slot_stride,
                         tile_cols=tile_cols, row_warps=row_warps, max_depth=max_depth)
    fn = load().gdn_verify_tree_prep if prep else load().gdn_verify_tree
    _check(fn(ctypes.byref(a), _ptr(parent), _ptr(depth_out), _stream(stream)),
           "gdn_verify_tree_prep" if prep else "gdn_verify_tree")


def gdn_commit_accepted(snapshots, accept_idx, state_cache, *, B, N, Hv, dk, dv, n_layers=1,
                        snap_layer_stride=0, cache_slot_stride=None, cache_layer_stride=0,
                        slot=None, n_slots=None, status=None, stream=None):
    """state_cache[l][slot[b]][h] = snapshots[l][b][accept_idx[b]][h] for every layer
    (fp32 snapshots; float16 ones go through gdn_commit_accepted_f16)."""
    if cache_slot_stride is None:
        cache_slot_stride = Hv * dk * dv
    if n_slots is None:
        n_slots = (state_cache.numel() - (n_layers - 1) * cache_layer_stride) // cache_slot_stride
    fn = load().gdn_commit_accepted
    name = "gdn_commit_accepted"
    if snapshots.dtype != state_cache.dtype:
        fn, name = load().gdn_commit_accepted_f16, "gdn_commit_accepted_f16"
    _check(fn(_ptr(snapshots), snap_layer_stride, _ptr(accept_idx), _ptr(state_cache),
              cache_slot_stride, cache_layer_stride, _ptr(slot), n_slots, B, N, Hv, dk, dv,
              n_layers, _ptr(status), _stream(stream)), name)


def gdn_commit_accepted_f16(snapshots_f16, accept_idx, state_cache, **kw):
    """gdn_commit_accepted from float16 snapshots, widened into the fp32 cache."""
    import torch

    _need(snapshots_f16.dtype == torch.float16, "snapshots_f16 must be float16")
    gdn_commit_accepted(snapshots_f16, accept_idx, state_cache, **kw)


def gdn_conv_commit(x, conv_state, accept_idx, *, parent=None, slot=None, n_slots=None,
                    state_slot_stride=None, status=None, stream=None):
    """Convolution-history commit in place: x [B,N,C] raw inputs of the block
    (bfloat16 or float32), conv_state [n_slots,C,W] of the same dtype; the
    history becomes the last W elements of [history, x of the accepted path]."""
    B, N, C = x.shape
    W = conv_state.shape[-1]
    _need(x.is_contiguous() and conv_state.is_contiguous(), "tensors must be contiguous")
    _need(x.dtype == conv_state.dtype, "x and conv_state must share a dtype")
    if state_slot_stride is None:
        state_slot_stride = C * W
    if n_slots is None:
        n_slots = conv_state.numel() // state_slot_stride
    _check(load().gdn_conv_commit(_ptr(x), _dtype_code(x), _ptr(conv_state), state_slot_stride,
                                  _ptr(slot), n_slots, _ptr(parent), _ptr(accept_idx), B, N, C,
                                  W, _ptr(status), _stream(stream)), "gdn_conv_commit")


def gdn_commit_index(accept_idx, slot, *, N, base_slot=0, status=None, stream=None):
    """Index-table commit: slot[b] = base_slot + b*N + accept_idx[b] (int32
    device tensors of B entries), so that the next verify reads its state from
    this block's snapshots buffer."""
    _need(accept_idx.is_contiguous() and slot.is_contiguous() and
          accept_idx.numel() == slot.numel(), "accept_idx and slot must be [B] int32")
    _check(load().gdn_commit_index(_ptr(accept_idx), accept_idx.numel(), N, base_slot, _ptr(slot),
                                   _ptr(status), _stream(stream)), "gdn_commit_index")


def gdn_replay_accepted(k, v, alpha, beta, state_cache, accept_idx, *, parent=None, slot=None,
                        n_slots=None, status=None, cache_slot_stride=None, tile_cols=0,
                        row_warps=0, stream=None, prep=False):
    """Checkpoint-and-replay commit: state_cache[slot[b]] <- the state of node
    accept_idx[b], recomputed over the accepted path from the cached state
    (chain when parent is None; parent [B,N] int32 for a tree)."""
    if parent is not None:
        _need(parent.is_contiguous() and tuple(parent.shape) == tuple(k.shape[:2]),
              "parent must be a contiguous [B,N] int32 tensor")
    _need(accept_idx.is_contiguous() and accept_idx.numel() == k.shape[0],
          "accept_idx must be a contiguous [B] int32 tensor")
    a = make_verify_args(None, k, v, alpha, beta, state_cache, None, None, slot=slot,
                         n_slots=n_slots, status=status, cache_slot_stride=cache_slot_stride,
                         tile_cols=tile_cols, row_warps=row_warps)
    fn = load().gdn_replay_accepted_prep if prep else load().gdn_replay_accepted
    _check(fn(ctypes.byref(a), _ptr(parent), _ptr(accept_idx), _stream(stream)),
           "gdn_replay_accepted_prep" if prep else "gdn_replay_accepted")


def gdn_prefill_workspace_bytes(T, Hk, Hv, dk, dv, chunk=64) -> int:
    return int(load().gdn_prefill_workspace_bytes(T, Hk, Hv, dk, dv, chunk))


def gdn_prefill_chunked(q, k, v, alpha, beta, state, o, workspace=None, *, chunk=64,
                        status=None, stream=None):
    """Chunked prefill of one sequence: q, k [T,Hk,dk]; v [T,Hv,dv]; alpha, beta [T,Hv];
    state [Hv,dk,dv] fp32 in/out; o [T,Hv,dv] fp32; workspace a uint8 device tensor of
    gdn_prefill_workspace_bytes(...) bytes (or None when that is 0); status an
    optional int32 device word that receives GDN_ERR_TIMEOUT if a bounded wait
    inside the kernel expired."""
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_prefill_chunked(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(alpha),
                                      _ptr(beta), T, Hk, Hv, dk, dv, chunk, _ptr(state), _ptr(o),
                                      _ptr(workspace), wbytes, _ptr(status), _stream(stream)),
           "gdn_prefill_chunked")


def gdn_prefill_chunked_noalloc(q, k, v, alpha, beta, state, o, *, chunk=64, status=None,
                                stream=None):
    """gdn_prefill_chunked on the library's built-in device scratch, for callers
    that cannot allocate device memory (no workspace argument).  Problems whose
    workspace would exceed PREFILL_NOALLOC_SCRATCH_BYTES raise GdnError with
    GDN_ERR_SCRATCH_LIMIT; calls that overlap on the GPU share the scratch and
    must be serialised by the caller."""
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    _check(load().gdn_prefill_chunked_noalloc(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q),
                                              _ptr(alpha), _ptr(beta), T, Hk, Hv, dk, dv, chunk,
                                              _ptr(state), _ptr(o), _ptr(status),
                                              _stream(stream)),
           "gdn_prefill_chunked_noalloc")


# ------------------------------------------------------- bound calls (serving)
class BoundCall:
    """One entry point with its arguments marshalled once.

    A serving loop that issues the same call every step (the same buffers,
    refilled in place) binds it once; each call then costs a single ctypes
    call: no shape checks, no argument struct built, no stream lookup.  The
    tensors given at binding time are kept alive by this object and must keep
    their addresses and shapes; the stream is fixed at binding time.  A
    non-zero status from the library raises GdnError, as the plain functions
    do."""

    __slots__ = ("_fn", "_name", "_args", "_keep")

    def __init__(self, fn, name, args, keep):
        self._fn, self._name, self._args, self._keep = fn, name, tuple(args), keep

    def __call__(self):
        code = self._fn(*self._args)
        if code != GDN_OK:
            raise GdnError(code, self._name)


def bind_verify_chain(q, k, v, alpha, beta, state_cache, snapshots, o, *, snapshots_f16=None,
                      stream=None, **kw):
    """gdn_verify_chain (or, with snapshots_f16, gdn_verify_chain_f16) bound
    to these buffers; keyword arguments as for gdn_verify_chain."""
    a = make_verify_args(q, k, v, alpha, beta, state_cache, snapshots, o, **kw)
    s = _stream(stream)
    if snapshots_f16 is not None:
        return BoundCall(load().gdn_verify_chain_f16, "gdn_verify_chain_f16",
                         (ctypes.byref(a), _ptr(snapshots_f16), s),
                         (a, q, k, v, alpha, beta, state_cache, snapshots_f16, o))
    return BoundCall(load().gdn_verify_chain, "gdn_verify_chain", (ctypes.byref(a), s),
                     (a, q, k, v, alpha, beta, state_cache, snapshots, o))


def bind_verify_tree(q, k, v, alpha, beta, state_cache, snapshots, o, parent, *, depth_out=None,
                     snapshots_f16=None, stream=None, **kw):
    """gdn_verify_tree (or, with snapshots_f16, gdn_verify_tree_f16) bound to
    these buffers; keyword arguments as for gdn_verify_tree."""
    _need(parent.is_contiguous() and tuple(parent.shape) == tuple(k.shape[:2]),
          "parent must be a contiguous [B,N] int32 tensor")
    a = make_verify_args(q, k, v, alpha, beta, state_cache, snapshots, o, **kw)
    s = _stream(stream)
    if snapshots_f16 is not None:
        return BoundCall(load().gdn_verify_tree_f16, "gdn_verify_tree_f16",
                         (ctypes.byref(a), _ptr(parent), _ptr(depth_out), _ptr(snapshots_f16), s),
                         (a, q, k, v, alpha, beta, state_cache, snapshots_f16, o, parent,
                          depth_out))
    return BoundCall(load().gdn_verify_tree, "gdn_verify_tree",
                     (ctypes.byref(a), _ptr(parent), _ptr(depth_out), s),
                     (a, q, k, v, alpha, beta, state_cache, snapshots, o, parent, depth_out))


def bind_commit_accepted(snapshots, accept_idx, state_cache, *, B, N, Hv, dk, dv, n_layers=1,
                         snap_layer_stride=0, cache_slot_stride=None, cache_layer_stride=0,
                         slot=None, n_slots=None, status=None, stream=None):
    """gdn_commit_accepted (gdn_commit_accepted_f16 for float16 snapshots)
    bound to these buffers."""
    if cache_slot_stride is None:
        cache_slot_stride = Hv * dk * dv
    if n_slots is None:
        n_slots = (state_cache.numel() - (n_layers - 1) * cache_layer_stride) // cache_slot_stride
    fn, name = load().gdn_commit_accepted, "gdn_commit_accepted"
    if snapshots.dtype != state_cache.dtype:
        fn, name = load().gdn_commit_accepted_f16, "gdn_commit_accepted_f16"
    args = (_ptr(snapshots), snap_layer_stride, _ptr(accept_idx), _ptr(state_cache),
            cache_slot_stride, cache_layer_stride, _ptr(slot), n_slots, B, N, Hv, dk, dv,
            n_layers, _ptr(status), _stream(stream))
    return BoundCall(fn, name, args, (snapshots, accept_idx, state_cache, slot, status))


def bind_replay_accepted(k, v, alpha, beta, state_cache, accept_idx, *, parent=None, stream=None,
                         **kw):
    """gdn_replay_accepted bound to these buffers."""
    a = make_verify_args(None, k, v, alpha, beta, state_cache, None, None, **kw)
    return BoundCall(load().gdn_replay_accepted, "gdn_replay_accepted",
                     (ctypes.byref(a), _ptr(parent), _ptr(accept_idx), _stream(stream)),
                     (a, k, v, alpha, beta, state_cache, accept_idx, parent))


def bind_prefill_chunked(q, k, v, alpha, beta, state, o, workspace=None, *, chunk=64,
                         status=None, stream=None):
    """gdn_prefill_chunked bound to these buffers."""
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(alpha), _ptr(beta), T, Hk, Hv, dk,
            dv, chunk, _ptr(state), _ptr(o), _ptr(workspace), wbytes, _ptr(status),
            _stream(stream))
    return BoundCall(load().gdn_prefill_chunked, "gdn_prefill_chunked", args,
                     (q, k, v, alpha, beta, state, o, workspace, status))
